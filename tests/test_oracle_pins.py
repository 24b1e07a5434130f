"""Pins for the CPU oracle: checks against facts fixed by the mathematics, not by the oracle.

The attention being pinned is the generalised PagedAttention of "Stateful
Large Language Model Serving with Pensieve" (abstract): several new query
tokens per request attend over that request's KV cache held in fixed-size,
non-contiguous blocks.  Each test below would fail for a plausible mistake in
the oracle: a wrong gather index (block / slot / head order), an off-by-one in
the causal mask, a missing scale, a wrong GQA head mapping, a sign error in the
max subtraction, or a wrong log base for LSE.

The independent route used here to read a request's logical K/V is block
indexing plus a reshape (``logical_kv``), not the oracle's per-key j // B, j % B
arithmetic.
"""
import json
import math
import os

import numpy as np
import pytest
import torch

import oracle
from paged_kv_attention_25_gb300 import workloads as wl

GOLDEN = os.path.join(os.path.dirname(__file__), "golden")


def f64(bits):
    return oracle.bf16_bits_to_f64(bits)


def logical_kv(pool, block_table_row, ctx):
    """[Hkv, ctx, D] logical view of one request: whole blocks stacked in table order."""
    nb = (ctx + pool.shape[2] - 1) // pool.shape[2]
    blocks = pool[block_table_row[:nb]]                  # [nb, Hkv, B, D]
    Hkv, B, D = blocks.shape[1:]
    return blocks.transpose(1, 0, 2, 3).reshape(Hkv, nb * B, D)[:, :ctx]


def dense_attention_fp64(qf, kf, vf, q_positions, scale):
    """Whole masked score matrix at once: rows at absolute positions q_positions."""
    s = scale * (qf @ kf.T)
    j = np.arange(kf.shape[0])[None, :]
    s = np.where(j > np.asarray(q_positions)[:, None], -np.inf, s)
    m = s.max(axis=1, keepdims=True)
    w = np.exp(s - m)
    l = w.sum(axis=1, keepdims=True)
    return (w @ vf) / l, (m + np.log(l))[:, 0]


def appended_pools(batch):
    kp, vp = batch.pool_arrays()
    oracle.append(kp, vp, batch.block_tables, batch.cu_q_lens, batch.q_positions, batch.k_new, batch.v_new)
    return kp, vp


def run_oracle(batch, kp, vp):
    return oracle.paged_attn(batch.q, kp, vp, batch.block_tables, batch.ctx_lens, batch.cu_q_lens,
                             batch.q_positions, batch.scale)


def brute_force(batch, kp, vp):
    T, Hq, D = batch.q.shape
    G = batch.num_q_heads // batch.num_kv_heads
    O = np.zeros((T, Hq, D))
    L = np.zeros((T, Hq))
    for r in range(batch.num_reqs):
        a, b = batch.cu_q_lens[r], batch.cu_q_lens[r + 1]
        if a == b:
            continue
        K = logical_kv(kp, batch.block_tables[r], batch.ctx_lens[r])
        V = logical_kv(vp, batch.block_tables[r], batch.ctx_lens[r])
        for h in range(Hq):
            o, l = dense_attention_fp64(f64(batch.q[a:b, h]), f64(K[h // G]), f64(V[h // G]),
                                        batch.q_positions[a:b], batch.scale)
            O[a:b, h] = o
            L[a:b, h] = l
    return O, L


@pytest.mark.parametrize("maker", [lambda: wl.tiny_mixed(1)] +
                         [(lambda s=s: wl.random_small(s)) for s in range(6)] +
                         [lambda: wl.random_small(11, num_q_heads=8, num_kv_heads=1, head_dim=32)])
def test_oracle_matches_dense_bruteforce(maker):
    batch = maker()
    kp, vp = appended_pools(batch)
    O, L = run_oracle(batch, kp, vp)
    Ob, Lb = brute_force(batch, kp, vp)
    np.testing.assert_allclose(O, Ob, rtol=1e-11, atol=1e-11)
    np.testing.assert_allclose(L, Lb, rtol=1e-11, atol=1e-11)


def test_append_read_back_and_canary():
    """After the append, each token's K/V sits at its logical position; nothing else changed."""
    batch = wl.random_small(3, num_q_heads=4, num_kv_heads=2)
    k0, v0 = batch.pool_arrays()
    kp, vp = k0.copy(), v0.copy()
    oracle.append(kp, vp, batch.block_tables, batch.cu_q_lens, batch.q_positions, batch.k_new, batch.v_new)
    written = np.zeros(kp.shape[:3], bool)               # [NB, Hkv, B]
    for r in range(batch.num_reqs):
        a, b = batch.cu_q_lens[r], batch.cu_q_lens[r + 1]
        Kl = logical_kv(kp, batch.block_tables[r], batch.ctx_lens[r])
        Vl = logical_kv(vp, batch.block_tables[r], batch.ctx_lens[r])
        for t in range(a, b):
            p = batch.q_positions[t]
            assert np.array_equal(Kl[:, p], batch.k_new[t])
            assert np.array_equal(Vl[:, p], batch.v_new[t])
        # mark the slots of this request's query positions through the same block-stack view
        nb = (batch.ctx_lens[r] + 15) // 16
        mark = np.zeros((nb * 16,), bool)
        mark[batch.q_positions[a:b]] = True
        for i in range(nb):
            written[batch.block_tables[r, i], :, :] |= mark[i * 16:(i + 1) * 16][None, :]
    assert np.array_equal(kp[~written], k0[~written])
    assert np.array_equal(vp[~written], v0[~written])
    assert written.sum() == batch.num_tokens * batch.num_kv_heads


def test_append_rejects_out_of_range_slot():
    batch = wl.tiny_mixed(1)
    kp, vp = batch.pool_arrays()
    bad = batch.q_positions.copy()
    bad[0] = batch.block_tables.shape[1] * 16            # beyond the block table
    before = kp.copy()
    with pytest.raises(ValueError):
        oracle.append(kp, vp, batch.block_tables, batch.cu_q_lens, bad, batch.k_new, batch.v_new)
    assert np.array_equal(kp, before)                     # nothing written


def test_attention_rejects_position_beyond_context():
    batch = wl.tiny_mixed(1)
    kp, vp = appended_pools(batch)
    pos = batch.q_positions.copy()
    pos[-1] = batch.ctx_lens[-1]                          # == ctx: not a valid key position
    with pytest.raises(ValueError):
        oracle.paged_attn(batch.q, kp, vp, batch.block_tables, batch.ctx_lens, batch.cu_q_lens, pos,
                          batch.scale)


def test_block_permutation_invariance_is_exact():
    """Moving physical blocks and rewriting the tables must not change a single bit."""
    batch = wl.random_small(7, num_q_heads=6, num_kv_heads=3)
    kp, vp = appended_pools(batch)
    O1, L1 = run_oracle(batch, kp, vp)
    rng = np.random.default_rng(123)
    perm = rng.permutation(batch.num_blocks)              # old id i -> new id perm[i]
    kp2 = np.empty_like(kp)
    vp2 = np.empty_like(vp)
    kp2[perm] = kp
    vp2[perm] = vp
    bt2 = np.where(batch.block_tables >= 0, perm[np.maximum(batch.block_tables, 0)], -1).astype(np.int32)
    O2, L2 = oracle.paged_attn(batch.q, kp2, vp2, bt2, batch.ctx_lens, batch.cu_q_lens,
                               batch.q_positions, batch.scale)
    assert np.array_equal(O1, O2) and np.array_equal(L1, L2)


def test_single_query_reduces_to_plain_decode():
    """q_len = 1 at the last position: softmax(scale * q K^T) V over the whole context."""
    reqs = [wl._decode(h) for h in (0, 15, 16, 17, 200)]
    batch = wl.build_batch("decode_pin", reqs, num_q_heads=2, num_kv_heads=2, head_dim=64, seed=21)
    kp, vp = appended_pools(batch)
    O, L = run_oracle(batch, kp, vp)
    for r in range(batch.num_reqs):
        K = f64(logical_kv(kp, batch.block_tables[r], batch.ctx_lens[r]))
        V = f64(logical_kv(vp, batch.block_tables[r], batch.ctx_lens[r]))
        for h in range(2):
            s = batch.scale * (K[h] @ f64(batch.q[r, h]))
            w = np.exp(s - s.max())
            np.testing.assert_allclose(O[r, h], (w @ V[h]) / w.sum(), rtol=1e-12, atol=1e-12)
            np.testing.assert_allclose(L[r, h], s.max() + math.log(w.sum()), rtol=1e-12, atol=1e-12)


def test_zero_context_is_causal_prefill_sdpa():
    """Pure prefill (no cached history) equals library causal attention (torch SDPA, fp64 CPU)."""
    reqs = [wl._new_turn(0, n) for n in (1, 7, 33)]
    batch = wl.build_batch("prefill_pin", reqs, num_q_heads=4, num_kv_heads=4, head_dim=64, seed=22)
    kp, vp = appended_pools(batch)
    O, L = run_oracle(batch, kp, vp)
    for r in range(batch.num_reqs):
        a, b = batch.cu_q_lens[r], batch.cu_q_lens[r + 1]
        q = torch.from_numpy(f64(batch.q[a:b]).transpose(1, 0, 2).copy())      # [H, n, D]
        k = torch.from_numpy(f64(batch.k_new[a:b]).transpose(1, 0, 2).copy())
        v = torch.from_numpy(f64(batch.v_new[a:b]).transpose(1, 0, 2).copy())
        o = torch.nn.functional.scaled_dot_product_attention(q, k, v, is_causal=True, scale=batch.scale)
        np.testing.assert_allclose(O[a:b], o.permute(1, 0, 2).numpy(), rtol=1e-10, atol=1e-10)
        s = batch.scale * (q @ k.transpose(1, 2))
        s = s.masked_fill(torch.triu(torch.ones(b - a, b - a, dtype=torch.bool), 1), float("-inf"))
        np.testing.assert_allclose(L[a:b], torch.logsumexp(s, -1).T.numpy(), rtol=1e-10, atol=1e-10)


def test_identical_keys_give_mean_of_visible_values():
    """k_j = k for every key: O[t] = mean of V[0..p_t], LSE = scale q.k + ln(p_t + 1)."""
    reqs = [wl._new_turn(20, 13), wl._recompute(40, 5, 3), wl._decode(31)]
    batch = wl.build_batch("identical_keys", reqs, num_q_heads=4, num_kv_heads=2, head_dim=64, seed=23)
    kp, vp = batch.pool_arrays()
    kvec = batch.k_new[0, 0].copy()
    kp[:] = kvec                                        # every slot, every head: the same key
    k_new = np.broadcast_to(kvec, batch.k_new.shape).copy()
    oracle.append(kp, vp, batch.block_tables, batch.cu_q_lens, batch.q_positions, k_new, batch.v_new)
    O, L = run_oracle(batch, kp, vp)
    G = 2
    for r in range(batch.num_reqs):
        V = f64(logical_kv(vp, batch.block_tables[r], batch.ctx_lens[r]))
        for t in range(batch.cu_q_lens[r], batch.cu_q_lens[r + 1]):
            p = batch.q_positions[t]
            for h in range(4):
                np.testing.assert_allclose(O[t, h], V[h // G, :p + 1].mean(axis=0), rtol=1e-12, atol=1e-12)
                s = batch.scale * float(f64(batch.q[t, h]) @ f64(kvec))
                assert abs(L[t, h] - (s + math.log(p + 1))) < 1e-12


def test_single_visible_key():
    """A query at position 0 sees one key: O = v_0, LSE = scale q.k_0."""
    reqs = [wl._new_turn(0, 1), wl._recompute(30, 1, 0)]
    batch = wl.build_batch("one_key", reqs, num_q_heads=2, num_kv_heads=1, head_dim=64, seed=24)
    kp, vp = appended_pools(batch)
    O, L = run_oracle(batch, kp, vp)
    for r in range(2):
        t = batch.cu_q_lens[r]
        K = f64(logical_kv(kp, batch.block_tables[r], batch.ctx_lens[r]))
        V = f64(logical_kv(vp, batch.block_tables[r], batch.ctx_lens[r]))
        for h in range(2):
            assert np.array_equal(O[t, h], V[0, 0])
            assert abs(L[t, h] - batch.scale * float(f64(batch.q[t, h]) @ K[0, 0])) < 1e-12


def test_gqa_equals_mha_with_repeated_kv_heads():
    """Grouped heads: query head h reads KV head h // G (contiguous groups)."""
    batch = wl.random_small(5, num_q_heads=8, num_kv_heads=2)
    kp, vp = appended_pools(batch)
    O, L = run_oracle(batch, kp, vp)
    kr = np.repeat(kp, 4, axis=1)
    vr = np.repeat(vp, 4, axis=1)
    O2, L2 = oracle.paged_attn(batch.q, kr, vr, batch.block_tables, batch.ctx_lens, batch.cu_q_lens,
                               batch.q_positions, batch.scale)
    assert np.array_equal(O, O2) and np.array_equal(L, L2)


def test_two_key_closed_form_golden():
    """Hand-derived two-key example (tests/golden/two_keys_closed_form.json)."""
    with open(os.path.join(GOLDEN, "two_keys_closed_form.json")) as f:
        g = json.load(f)
    D = 64
    B = 16

    def vec(vals):
        x = np.zeros(D, np.float32)
        x[:len(vals)] = vals
        return wl.f32_to_bf16_bits(x)

    kp = np.zeros((2, 1, B, D), np.uint16)
    vp = np.zeros((2, 1, B, D), np.uint16)
    kp[1, 0, 0] = vec(g["k0"])
    kp[1, 0, 1] = vec(g["k1"])
    vp[1, 0, 0] = vec(g["v0"])
    vp[1, 0, 1] = vec(g["v1"])
    q = vec(g["q"]).reshape(1, 1, D)
    O, L = oracle.paged_attn(q, kp, vp, np.array([[1]], np.int32), np.array([2], np.int32),
                             np.array([0, 1], np.int32), np.array([1], np.int32), g["scale"])
    np.testing.assert_allclose(O[0, 0, :2], g["expected_o"], rtol=0, atol=1e-14)
    assert abs(L[0, 0] - g["expected_lse"]) < 1e-14


def test_tiny_mixed_regression_fixture():
    """Oracle output on the tiny workload, stored by tests/golden/make_golden.py."""
    with open(os.path.join(GOLDEN, "tiny_mixed_oracle.json")) as f:
        g = json.load(f)
    batch = wl.tiny_mixed(g["seed"])
    kp, vp = appended_pools(batch)
    O, L = run_oracle(batch, kp, vp)
    np.testing.assert_allclose(L, np.array(g["lse"]), rtol=0, atol=1e-12)
    np.testing.assert_allclose(O.sum(axis=2), np.array(g["o_row_sums"]), rtol=0, atol=1e-10)


def test_swap_roundtrip_moves_whole_blocks():
    batch = wl.random_small(2)
    kp, vp = appended_pools(batch)
    ids = batch.used_blocks[:5]
    host = oracle.swap_out(kp, vp, ids)
    assert np.array_equal(host[:, 0], kp[ids]) and np.array_equal(host[:, 1], vp[ids])
    free = np.setdiff1d(np.arange(batch.num_blocks), batch.used_blocks)[:5]
    k2, v2 = kp.copy(), vp.copy()
    oracle.swap_in(k2, v2, free, host)
    assert np.array_equal(k2[free], kp[ids]) and np.array_equal(v2[free], vp[ids])
    others = np.setdiff1d(np.arange(batch.num_blocks), free)
    assert np.array_equal(k2[others], kp[others])
    with pytest.raises(ValueError):
        oracle.swap_out(kp, vp, np.array([batch.num_blocks], np.int32))


# ----------------------------------------------------------------------------- FP8 (E4M3) KV cache
# The codec is pinned to torch's float8_e4m3fn conversions (a library routine
# for the same format) and to a brute-force nearest-code search; the FP8
# attention and append are pinned to the (already pinned) bf16 oracle on values
# that both formats hold exactly.

def _e4m3_table():
    vals = oracle.e4m3_decode(np.arange(256, dtype=np.uint8))
    return np.arange(256), vals


def test_e4m3_decode_matches_torch_for_every_code():
    codes = np.arange(256, dtype=np.uint8)
    ours = oracle.e4m3_decode(codes)
    ref = torch.from_numpy(codes).view(torch.float8_e4m3fn).to(torch.float64).numpy()
    assert np.array_equal(np.isnan(ours), np.isnan(ref)) and np.isnan(ours).sum() == 2   # 0x7F, 0xFF
    ok = ~np.isnan(ref)
    assert np.array_equal(ours[ok], ref[ok])
    assert ours[0x7E] == 448.0 and ours[0x38] == 1.0 and ours[0x01] == 2.0 ** -9 and ours[0x08] == 2.0 ** -6


def test_e4m3_encode_matches_torch_within_range():
    rng = np.random.default_rng(5)
    x = np.concatenate([rng.standard_normal(40000) * 60, rng.standard_normal(20000) * 2.0 ** -7,
                        rng.uniform(-447.9, 447.9, 20000)]).astype(np.float32)
    _, vals = _e4m3_table()
    pos = np.unique(vals[(vals > 0) & ~np.isnan(vals)])
    mids = ((pos[:-1] + pos[1:]) / 2).astype(np.float32)          # exact ties, both signs
    x = np.concatenate([x, mids, -mids, np.float32([0.0, -0.0])])
    ours = oracle.e4m3_encode(x)
    ref = torch.from_numpy(x).to(torch.float8_e4m3fn).view(torch.uint8).numpy()
    assert np.array_equal(ours, ref)


def test_e4m3_encode_is_nearest_code_with_ties_to_even():
    codes, vals = _e4m3_table()
    fin = ~np.isnan(vals)
    codes, vals = codes[fin], vals[fin]
    rng = np.random.default_rng(6)
    pos = np.unique(vals[vals > 0])
    mids = (pos[:-1] + pos[1:]) / 2
    x = np.concatenate([rng.uniform(-600, 600, 3000), rng.uniform(-2.0 ** -5, 2.0 ** -5, 2000), mids, -mids,
                        [448.0, 455.0, 464.0, 1000.0, -1000.0]]).astype(np.float32)
    got = oracle.e4m3_encode(x)
    for xi, gi in zip(x.astype(np.float64), got):
        d = np.abs(vals - xi)
        cand = codes[d == d.min()]
        cand = cand[(cand >> 7) == (1 if np.signbit(xi) else 0)] if len(cand) > 1 else cand
        if len(cand) > 1:   # a tie between neighbours: the even mantissa wins
            cand = cand[(cand & 1) == 0]
        assert len(cand) == 1 and gi == cand[0], (xi, gi, cand)


def test_e4m3_encode_saturates_and_keeps_nan():
    got = oracle.e4m3_encode(np.float32([1e6, -1e6, np.inf, -np.inf, 449.0, -463.9]))
    assert list(got) == [0x7E, 0xFE, 0x7E, 0xFE, 0x7E, 0xFE]
    nan_code = int(oracle.e4m3_encode(np.float32([np.nan]))[0])
    assert nan_code & 0x7F == 0x7F


def _exact_e4m3_bf16(shape, rng):
    """bf16 bit patterns of values that E4M3 holds exactly (|v| in [2^-6, 240])."""
    codes = rng.integers(0, 112, size=shape)
    codes = ((codes // 56) << 7) | ((1 + (codes % 56) // 8 * 2) << 3) | (codes % 8)
    vals = oracle.e4m3_decode(codes.astype(np.uint8)).astype(np.float32)
    return (vals.view(np.uint32) >> 16).astype(np.uint16)


def test_fp8_append_equals_bf16_append_on_exact_values():
    # scale 1 and values that E4M3 holds exactly: every code decodes to the
    # appended value, in the slot the bf16 append writes.
    b = wl.random_small(31, num_q_heads=4, num_kv_heads=2, head_dim=64)
    rng = np.random.default_rng(31)
    kn, vn = _exact_e4m3_bf16(b.k_new.shape, rng), _exact_e4m3_bf16(b.v_new.shape, rng)
    shape = (b.num_blocks, 2, 16, 64)
    k8, v8 = np.zeros(shape, np.uint8), np.zeros(shape, np.uint8)
    oracle.append_fp8(k8, v8, 1.0, 1.0, b.block_tables, b.cu_q_lens, b.q_positions, kn, vn)
    kb, vb = np.zeros(shape, np.uint16), np.zeros(shape, np.uint16)
    oracle.append(kb, vb, b.block_tables, b.cu_q_lens, b.q_positions, kn, vn)
    assert np.array_equal(oracle.e4m3_decode(k8), f64(kb)) and np.array_equal(oracle.e4m3_decode(v8), f64(vb))


def test_fp8_append_rounds_each_quotient_to_its_nearest_code():
    b = wl.random_small(32, num_q_heads=4, num_kv_heads=2, head_dim=64)
    ks, vs = np.float32(0.0123), np.float32(0.5)
    shape = (b.num_blocks, 2, 16, 64)
    k8, v8 = np.zeros(shape, np.uint8), np.zeros(shape, np.uint8)
    oracle.append_fp8(k8, v8, ks, vs, b.block_tables, b.cu_q_lens, b.q_positions, b.k_new, b.v_new)
    kb = np.zeros(shape, np.uint16)
    oracle.append(kb, np.zeros(shape, np.uint16), b.block_tables, b.cu_q_lens, b.q_positions, b.k_new, b.v_new)
    mark = np.zeros(shape, np.uint16)
    oracle.append(mark, np.zeros(shape, np.uint16), b.block_tables, b.cu_q_lens, b.q_positions,
                  np.full_like(b.k_new, 0x3F80), np.full_like(b.v_new, 0x3F80))   # 1.0 in every written slot
    written = mark != 0
    x = (f64(kb[written]).astype(np.float32) / ks).astype(np.float64)
    got = oracle.e4m3_decode(k8[written])
    _, vals = _e4m3_table()
    fin = np.sort(vals[~np.isnan(vals)])
    # |code value - quotient| is the distance to the nearest representable value (saturating at 448)
    nearest = np.abs(fin[None, :] - np.clip(x, -448, 448)[:, None]).min(axis=1)
    assert np.allclose(np.abs(got - np.clip(x, -448, 448)), nearest, rtol=0, atol=0)
    assert (k8[~written] == 0).all() and (v8[~written] == 0).all()


def test_fp8_attention_equals_bf16_attention_on_exact_values():
    # Power-of-two scales: every dequantised value is a bf16 value, so the FP8
    # oracle must reproduce the bf16 oracle on the equivalent bf16 pools.
    b = wl.decode_small(33, num_q_heads=8, num_kv_heads=4, head_dim=64, num_reqs=4, max_ctx=200)
    k8, v8 = wl.fp8_pool_arrays(b)
    ks, vs = 2.0 ** -6, 2.0 ** -4
    to_bf16 = lambda codes, s: ((oracle.e4m3_decode(codes) * s).astype(np.float32).view(np.uint32) >> 16).astype(np.uint16)
    kb, vb = to_bf16(k8, ks), to_bf16(v8, vs)
    assert np.array_equal(f64(kb), oracle.e4m3_decode(k8) * ks)
    O8, L8 = oracle.paged_attn_fp8(b.q, k8, v8, ks, vs, b.block_tables, b.ctx_lens, b.cu_q_lens, b.q_positions, b.scale)
    O, L = oracle.paged_attn(b.q, kb, vb, b.block_tables, b.ctx_lens, b.cu_q_lens, b.q_positions, b.scale)
    assert np.allclose(O8, O, rtol=0, atol=1e-12) and np.allclose(L8, L, rtol=0, atol=1e-12)
