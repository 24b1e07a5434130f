"""CPU-only checks of the C ABI: the library builds, loads without a GPU, exports
every symbol include/pkv.h declares, plans batches correctly on the host, and
reports errors instead of crashing when no device is present."""
import ctypes
import os
import re

import numpy as np
import pytest
import torch

from paged_kv_attention_25_gb300 import build as pkv_build
from paged_kv_attention_25_gb300 import pkv
from paged_kv_attention_25_gb300 import workloads as wl

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


@pytest.fixture(scope="module")
def lib():
    pkv_build.build()
    return pkv.load_library()


def header_functions():
    with open(os.path.join(ROOT, "include", "pkv.h")) as f:
        text = f.read()
    text = re.sub(r"/\*.*?\*/", "", text, flags=re.S)
    return sorted(set(re.findall(r"\b(pkv_[a-z_0-9]+)\s*\(", text)))


def test_library_exports_every_declared_symbol(lib):
    names = header_functions()
    assert len(names) >= 16
    for n in names:
        assert hasattr(lib, n), f"{n} declared in include/pkv.h but not exported"
    assert sorted(pkv.EXPORTED) == names


def test_version_and_error_string(lib):
    assert "sm_103a" in pkv.pkv_version()
    assert isinstance(pkv.pkv_last_error(), str)


@pytest.mark.skipif(torch.cuda.is_available(), reason="checks the no-device path")
def test_calls_without_device_fail_cleanly(lib):
    desc = pkv.pkv_pool_desc(64, 16, 4, 64, 0, None, None)
    h = ctypes.c_void_p()
    rc = lib.pkv_pool_create(ctypes.byref(desc), ctypes.byref(h))
    assert rc in (pkv.PKV_ECUDA, pkv.PKV_ENOMEM)
    assert pkv.pkv_last_error() != ""
    assert not h.value


def test_swap_in_ahead_rejects_null_pool(lib):
    ids = (ctypes.c_int32 * 1)(0)
    buf = ctypes.create_string_buffer(64)
    assert lib.pkv_swap_in_ahead(None, ids, 1, buf, None, None) == pkv.PKV_EINVAL
    assert lib.pkv_swap_in_finish(None, None) == pkv.PKV_EINVAL
    assert "pool" in pkv.pkv_last_error()


def test_pool_create_rejects_bad_shapes(lib):
    for desc, code in [(pkv.pkv_pool_desc(64, 32, 4, 64, 0, None, None), pkv.PKV_EUNSUPPORTED),
                       (pkv.pkv_pool_desc(64, 16, 4, 96, 0, None, None), pkv.PKV_EUNSUPPORTED),
                       (pkv.pkv_pool_desc(0, 16, 4, 64, 0, None, None), pkv.PKV_EINVAL),
                       (pkv.pkv_pool_desc(64, 16, 4, 64, 7, None, None), pkv.PKV_EUNSUPPORTED),
                       # FP8 pools need finite positive scales (checked before any CUDA call)
                       (pkv.pkv_pool_desc(64, 16, 4, 64, pkv.PKV_DTYPE_FP8_E4M3, None, None, 0.0, 1.0), pkv.PKV_EINVAL),
                       (pkv.pkv_pool_desc(64, 16, 4, 64, pkv.PKV_DTYPE_FP8_E4M3, None, None, 1.0, -2.0), pkv.PKV_EINVAL),
                       (pkv.pkv_pool_desc(64, 16, 4, 64, pkv.PKV_DTYPE_FP8_E4M3, None, None, float("nan"), 1.0),
                        pkv.PKV_EINVAL),
                       (pkv.pkv_pool_desc(64, 16, 4, 64, pkv.PKV_DTYPE_FP8_E4M3, None, None, float("inf"), 1.0),
                        pkv.PKV_EINVAL)]:
        h = ctypes.c_void_p()
        assert lib.pkv_pool_create(ctypes.byref(desc), ctypes.byref(h)) == code


def check_plan(batch, num_sms=148):
    meta = pkv.HostMeta(batch.cu_q_lens, batch.ctx_lens, batch.q_positions)
    Hq, Hkv, D = batch.num_q_heads, batch.num_kv_heads, batch.head_dim
    G = Hq // Hkv
    items, st = pkv.pkv_plan_inspect(Hq, Hkv, D, num_sms, meta)
    # Split-KV items run longest first.  Tensor-core items run one request
    # after another (a request's tile pairs share its K/V in L2): each
    # request's items are contiguous and longest first, and requests follow
    # the order of their longest items.
    lens = [int(it["kv_end"]) - int(it["kv_start"]) for it in items if int(it["kernel"]) == 1]
    assert all(a >= b for a, b in zip(lens, lens[1:])), "split-KV items not longest first"
    tc = [(int(it["req"]), int(it["kv_end"]) - int(it["kv_start"])) for it in items if int(it["kernel"]) == 2]
    runs = []
    for r, n in tc:
        if runs and runs[-1][0] == r:
            assert runs[-1][1][-1] >= n, "tensor-core items of a request not longest first"
            runs[-1][1].append(n)
        else:
            assert all(rr != r for rr, _ in runs), "tensor-core items of a request not contiguous"
            runs.append((r, [n]))
    heads = [ns[0] for _, ns in runs]
    assert all(a >= b for a, b in zip(heads, heads[1:])), "requests not ordered by their longest item"
    # Group items by (kernel, request, kv head, q_start, q_count).
    groups = {}
    for it in items:
        key = (int(it["req"]), int(it["kv_head"]), int(it["q_start"]), int(it["q_count"]) + int(it["q_count2"]))
        if int(it["kernel"]) == 1:
            assert int(it["q_count2"]) == 0
        else:
            assert int(it["q_count"]) * G <= 128 and int(it["q_count2"]) * G <= 128
        groups.setdefault(key, []).append(it)
        # position bounds of each tile: exact, since the host knows the positions
        q0, c0, c1 = int(it["q_start"]), int(it["q_count"]), int(it["q_count2"])
        for t0, c, mx, mn in ((q0, c0, it["pos_max0"], it["pos_min0"]), (q0 + c0, c1, it["pos_max1"], it["pos_min1"])):
            if c == 0:
                assert int(mx) == -1
            else:
                assert int(mx) == int(batch.q_positions[t0:t0 + c].max())
                assert int(mn) == int(batch.q_positions[t0:t0 + c].min())
    covered = np.zeros((batch.num_tokens, Hkv), np.int32)
    part_rows = []
    dec_bytes = tc_bytes = 0
    for (r, g, q0, qc), its in groups.items():
        kernels = {int(i["kernel"]) for i in its}
        assert len(kernels) == 1
        kern = kernels.pop()
        rows = qc * G
        if kern == 1:
            assert rows <= 4
        else:
            assert rows <= 256
        a, b = batch.cu_q_lens[r], batch.cu_q_lens[r + 1]
        assert a <= q0 and q0 + qc <= b
        covered[q0:q0 + qc, g] += 1
        kv_len = min(int(batch.ctx_lens[r]), int(batch.q_positions[q0:q0 + qc].max()) + 1)
        its = sorted(its, key=lambda i: int(i["kv_start"]))
        unit = 16 if kern == 1 else 128
        # splits tile [0, kv_len) exactly, in whole units
        assert int(its[0]["kv_start"]) == 0 and int(its[-1]["kv_end"]) == kv_len
        for x, y in zip(its[:-1], its[1:]):
            assert int(x["kv_end"]) == int(y["kv_start"])
        for i in its:
            assert int(i["kv_start"]) % unit == 0 and int(i["kv_end"]) > int(i["kv_start"])
        if len(its) == 1:
            assert int(its[0]["part"]) == -1
        else:
            for i in its:
                assert int(i["part"]) >= 0
                part_rows.append((int(i["part"]), rows))
    assert np.all(covered == 1), "every (token, KV head) in exactly one query group"
    # partial rows do not overlap
    part_rows.sort()
    for (p0, n0), (p1, _) in zip(part_rows[:-1], part_rows[1:]):
        assert p0 + n0 <= p1
    assert st["num_partial_rows"] == (part_rows[-1][0] + part_rows[-1][1] if part_rows else 0)
    # algorithmic KV bytes: each request's visible keys once, all KV heads, K and V
    tot = 0
    for r in range(batch.num_reqs):
        a, b = batch.cu_q_lens[r], batch.cu_q_lens[r + 1]
        if a < b:
            tot += min(int(batch.ctx_lens[r]), int(batch.q_positions[a:b].max()) + 1) * 4 * Hkv * D
    assert st["decode_kv_bytes"] + st["tc_kv_bytes"] == tot
    return items, st


@pytest.mark.parametrize("maker", [lambda: wl.tiny_mixed(1), lambda: wl.random_small(3),
                                   lambda: wl.random_small(4, num_q_heads=8, num_kv_heads=1),
                                   lambda: wl.random_small(9, num_q_heads=16, num_kv_heads=2, max_ctx=3000,
                                                           max_q=300)])
def test_planner_covers_every_row_once(lib, maker):
    check_plan(maker())


def test_planner_random_batches(lib):
    # Random shapes, lengths and request mixes (decode, prefill, new turn, recompute),
    # and SM counts from one SM up, through the same coverage and ordering checks.
    rng = np.random.default_rng(2024)
    for seed in range(40):
        g = int(rng.choice([1, 2, 4, 5, 8]))
        hkv = int(rng.integers(1, 5))
        b = wl.random_small(100 + seed, num_q_heads=g * hkv, num_kv_heads=hkv, head_dim=int(rng.choice([64, 128])),
                            num_reqs=int(rng.integers(1, 9)), max_ctx=int(rng.integers(2, 2500)),
                            max_q=int(rng.integers(1, 200)))
        check_plan(b, num_sms=int(rng.choice([1, 7, 148, 152])))


def test_planner_splits_long_context_and_routes(lib):
    """One 65,537-token decode next to short requests: the long one is cut into many splits."""
    reqs = [wl._decode(65536), wl._decode(100), wl._new_turn(50, 30),
            wl._recompute(900, 100, 40)]
    batch = wl.build_batch("skew", reqs, num_q_heads=8, num_kv_heads=8, head_dim=128, seed=3)
    items, st = check_plan(batch, num_sms=152)
    long_items = items[(items["req"] == 0)]
    assert len(long_items) > 8 * 8        # > 8 splits per KV head
    assert set(items[items["req"] == 2]["kernel"]) == {2}   # 30-token new turn -> tensor cores
    assert set(items[items["req"] == 1]["kernel"]) == {1}   # single decode token -> split-KV
    # recompute request: tiles stop at the position jump between [0,100) and [900,940)
    rq = items[items["req"] == 3]
    assert all(not (q0 < 100 < q0 + qc) for q0, qc in zip(rq["q_start"] - batch.cu_q_lens[3], rq["q_count"]))


@pytest.mark.parametrize("name", ["llama13b_mixed", "llama70b_gqa", "long_skewed_evict"])
def test_planner_on_full_workload_shapes(lib, name):
    batch = {"llama13b_mixed": wl.llama13b_mixed, "llama70b_gqa": wl.llama70b_gqa,
             "long_skewed_evict": wl.long_skewed_evict}[name]()
    items, st = check_plan(batch, num_sms=152)
    assert st["num_decode_items"] + st["num_tc_items"] == len(items)


def test_planner_rejects_bad_metadata(lib):
    b = wl.tiny_mixed(1)
    bad = b.q_positions.copy()
    bad[0] = b.ctx_lens[0]
    with pytest.raises(pkv.PkvError):
        pkv.pkv_plan_inspect(4, 4, 64, 148, pkv.HostMeta(b.cu_q_lens, b.ctx_lens, bad))
    cu = b.cu_q_lens.copy()
    cu[0] = 1
    with pytest.raises(pkv.PkvError):
        pkv.pkv_plan_inspect(4, 4, 64, 148, pkv.HostMeta(cu, b.ctx_lens, b.q_positions))
    with pytest.raises(pkv.PkvError):
        pkv.pkv_plan_inspect(6, 4, 64, 148, pkv.HostMeta(b.cu_q_lens, b.ctx_lens, b.q_positions))


def test_planner_without_host_positions_covers_whole_context(lib):
    b = wl.random_small(6)
    meta = pkv.HostMeta(b.cu_q_lens, b.ctx_lens, None)
    items, _ = pkv.pkv_plan_inspect(b.num_q_heads, b.num_kv_heads, b.head_dim, 148, meta)
    for r in range(b.num_reqs):
        its = items[items["req"] == r]
        if len(its):
            assert its["kv_end"].max() == b.ctx_lens[r]
            # unknown positions: bounds cover the whole context
            assert (its["pos_max0"] == b.ctx_lens[r] - 1).all() and (its["pos_min0"] == 0).all()


def _expected_decode_items(batch, num_sms):
    """Split-KV item count under the planner's rule: the smallest of 1..4 splits per
    CTA slot (3 per SM) whose items fill two waves, else 4; chunks in 16-key blocks,
    at least 16 blocks, an even split of each (request, KV head) key range."""
    G = batch.num_q_heads // batch.num_kv_heads
    groups = []
    for r in range(batch.num_reqs):
        a, b = int(batch.cu_q_lens[r]), int(batch.cu_q_lens[r + 1])
        if a < b and (b - a) * G <= 4:
            kv = min(int(batch.ctx_lens[r]), int(batch.q_positions[a:b].max()) + 1)
            groups.append(-(-kv // 16))
    if not groups:
        return 0
    slots = num_sms * 3
    total = sum(groups) * batch.num_kv_heads

    def items(chunk):
        n = 0
        for u in groups:
            per = -(-u // max(1, -(-u // chunk)))
            n += max(1, -(-u // per))
        return n * batch.num_kv_heads

    chunk_for = lambda s: max(16, -(-total // (slots * s)))
    for s in (1, 2, 3):
        if items(chunk_for(s)) >= 2 * slots:
            return items(chunk_for(s))
    return items(chunk_for(4))


@pytest.mark.parametrize("name", ["llama13b_mixed", "long_skewed_evict", "decode_lognormal_small"])
def test_split_kv_split_count_fills_two_waves(lib, name):
    batch = wl.WORKLOADS[name]()
    meta = pkv.HostMeta(batch.cu_q_lens, batch.ctx_lens, batch.q_positions)
    _, st = pkv.pkv_plan_inspect(batch.num_q_heads, batch.num_kv_heads, batch.head_dim, 152, meta)
    assert st["num_decode_items"] == _expected_decode_items(batch, 152)
    # the headline mix needs no split at all; the 65,536-token request still splits
    if name == "llama13b_mixed":
        assert st["num_merge_items"] == 0
    if name == "long_skewed_evict":
        assert st["num_decode_items"] >= 2 * 152 * 3 and st["num_merge_items"] > 0
