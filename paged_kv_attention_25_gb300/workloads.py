"""Seeded synthetic input generators for paged multi-token attention.

This module only *draws inputs*: request shapes, block tables, pool contents,
queries and new keys/values.  It holds none of the attention arithmetic and
none of the paging index math beyond choosing which physical blocks a request
owns, so both the CUDA path and the CPU oracle can consume what it produces.

Workload shapes follow the multi-turn serving setting of "Stateful Large
Language Model Serving with Pensieve" (abstract: a conversation's cached
history plus several new input tokens per request, cache spread over
non-contiguous GPU memory), with Llama-2-13B (40 MHA heads, head_dim 128) and
Llama-2-70B (64 query / 8 KV heads) attention-layer shapes.  The real
conversation datasets are not available, so every workload is synthetic:
values are N(0,1) drawn in fp32 and rounded once to bf16 (round to nearest
even), and physical block ids are a seeded random permutation of the pool so
that every request's blocks are scattered.

A request is described by its context length ``ctx`` (keys visible after this
step's append) and its query positions (absolute positions, unique, each
``< ctx``).  Positions in ``[0, ctx)`` that are not query positions are
"cached history" and are present in the pool before the step; query
positions receive their K/V through the append.
"""
from __future__ import annotations

import math
import os
from concurrent.futures import ThreadPoolExecutor
from dataclasses import dataclass, field

import numpy as np

BLOCK_SIZE = 16


def f32_to_bf16_bits(x: np.ndarray) -> np.ndarray:
    """Round fp32 values to bf16 (round to nearest, ties to even); return raw uint16 bits.

    Inputs here are finite normals, so NaN handling is not needed.
    """
    u = np.ascontiguousarray(x, dtype=np.float32).view(np.uint32)
    bias = ((u >> 16) & np.uint32(1)) + np.uint32(0x7FFF)
    return ((u + bias) >> 16).astype(np.uint16)


def _normal_bf16(seed_seq: np.random.SeedSequence, shape, chunk_rows: int | None = None) -> np.ndarray:
    """N(0,1) bf16 bits of the given shape, drawn in independent chunks along axis 0.

    Each chunk has its own child SeedSequence, so the result does not depend on
    how many threads draw it.
    """
    shape = tuple(int(s) for s in shape)
    out = np.empty(shape, dtype=np.uint16)
    n0 = shape[0]
    if n0 == 0:
        return out
    per_row = int(np.prod(shape[1:])) if len(shape) > 1 else 1
    if chunk_rows is None:
        chunk_rows = max(1, (1 << 22) // max(per_row, 1))
    starts = list(range(0, n0, chunk_rows))
    children = seed_seq.spawn(len(starts))

    def fill(i):
        s = starts[i]
        e = min(n0, s + chunk_rows)
        g = np.random.Generator(np.random.PCG64(children[i]))
        vals = g.standard_normal((e - s,) + shape[1:], dtype=np.float32)
        out[s:e] = f32_to_bf16_bits(vals)

    workers = min(len(starts), os.cpu_count() or 1, 32)
    if workers <= 1:
        for i in range(len(starts)):
            fill(i)
    else:
        with ThreadPoolExecutor(workers) as ex:
            list(ex.map(fill, range(len(starts))))
    return out


@dataclass
class RequestSpec:
    """One request of a unified batch: context length and absolute query positions."""
    ctx: int
    q_positions: np.ndarray  # int32, unique, each < ctx
    kind: str = "mixed"      # "decode", "prefill", "new_turn", "recompute" (labels only)


@dataclass
class Batch:
    """A fully materialised synthetic batch (all arrays are numpy, host side).

    Layouts:
      q          [T, Hq, D]        bf16 bits (uint16)
      k_new,v_new[T, Hkv, D]       bf16 bits, K/V of the T query tokens (appended this step)
      block_tables [R, max_blocks] int32, -1 padded
      ctx_lens   [R] int32, cu_q_lens [R+1] int32, q_positions [T] int32
      used_blocks [U] int32 (sorted physical ids referenced by some block table)
      k_used,v_used [U, Hkv, B, D] bf16 bits: pool contents of those blocks before the step
    Blocks of the pool that no request references hold zeros.
    """
    name: str
    num_q_heads: int
    num_kv_heads: int
    head_dim: int
    block_size: int
    num_blocks: int
    scale: float
    ctx_lens: np.ndarray
    cu_q_lens: np.ndarray
    q_positions: np.ndarray
    block_tables: np.ndarray
    q: np.ndarray
    k_new: np.ndarray
    v_new: np.ndarray
    used_blocks: np.ndarray
    k_used: np.ndarray
    v_used: np.ndarray
    kinds: list = field(default_factory=list)
    seed: int = 0

    @property
    def num_reqs(self) -> int:
        return int(self.ctx_lens.shape[0])

    @property
    def num_tokens(self) -> int:
        return int(self.q_positions.shape[0])

    @property
    def max_blocks(self) -> int:
        return int(self.block_tables.shape[1])

    def pool_arrays(self):
        """Full-size host pools [NB, Hkv, B, D] (zeros except the used blocks)."""
        shp = (self.num_blocks, self.num_kv_heads, self.block_size, self.head_dim)
        kp = np.zeros(shp, dtype=np.uint16)
        vp = np.zeros(shp, dtype=np.uint16)
        kp[self.used_blocks] = self.k_used
        vp[self.used_blocks] = self.v_used
        return kp, vp

    def kv_bytes_per_elem(self) -> int:
        return 2

    def describe(self) -> dict:
        q_lens = np.diff(self.cu_q_lens)
        return {
            "workload": self.name,
            "num_reqs": self.num_reqs,
            "num_q_tokens": self.num_tokens,
            "num_q_heads": self.num_q_heads,
            "num_kv_heads": self.num_kv_heads,
            "head_dim": self.head_dim,
            "block_size": self.block_size,
            "pool_blocks": self.num_blocks,
            "ctx_total": int(self.ctx_lens.sum()),
            "ctx_max": int(self.ctx_lens.max()) if self.num_reqs else 0,
            "q_len_max": int(q_lens.max()) if self.num_reqs else 0,
            "seed": self.seed,
        }


def build_batch(name: str, requests: list[RequestSpec], *, num_q_heads: int, num_kv_heads: int,
                head_dim: int, block_size: int = BLOCK_SIZE, num_blocks: int | None = None,
                pool_factor: float = 1.25, seed: int = 0, scale: float | None = None) -> Batch:
    """Materialise a batch: scattered block tables, pool contents and Q / new K, V.

    ``num_blocks`` defaults to ``ceil(pool_factor * blocks_needed)``.  Physical
    ids are handed out from one seeded random permutation of the pool.
    """
    ss = np.random.SeedSequence(seed)
    s_perm, s_pool_k, s_pool_v, s_q, s_kn, s_vn = ss.spawn(6)
    R = len(requests)
    ctx = np.array([r.ctx for r in requests], dtype=np.int32)
    nblk = [(int(c) + block_size - 1) // block_size for c in ctx]
    need = int(sum(nblk))
    if num_blocks is None:
        num_blocks = max(need, int(math.ceil(pool_factor * need)), 1)
    if need > num_blocks:
        raise ValueError(f"pool of {num_blocks} blocks cannot hold {need}")
    perm = np.random.Generator(np.random.PCG64(s_perm)).permutation(num_blocks).astype(np.int32)
    max_blocks = max(nblk) if nblk else 1
    max_blocks = max(max_blocks, 1)
    bt = np.full((R, max_blocks), -1, dtype=np.int32)
    off = 0
    for i, nb in enumerate(nblk):
        bt[i, :nb] = perm[off:off + nb]
        off += nb
    qpos = []
    cu = [0]
    for r in requests:
        p = np.asarray(r.q_positions, dtype=np.int32)
        if p.size and (p.min() < 0 or p.max() >= r.ctx):
            raise ValueError("query position outside [0, ctx)")
        if np.unique(p).size != p.size:
            raise ValueError("duplicate query position")
        qpos.append(p)
        cu.append(cu[-1] + p.size)
    q_positions = np.concatenate(qpos).astype(np.int32) if qpos else np.zeros(0, np.int32)
    T = int(cu[-1])
    used = np.sort(perm[:need]).astype(np.int32)
    shp = (need, num_kv_heads, block_size, head_dim)
    k_used = _normal_bf16(s_pool_k, shp)
    v_used = _normal_bf16(s_pool_v, shp)
    q = _normal_bf16(s_q, (T, num_q_heads, head_dim))
    k_new = _normal_bf16(s_kn, (T, num_kv_heads, head_dim))
    v_new = _normal_bf16(s_vn, (T, num_kv_heads, head_dim))
    if scale is None:
        scale = 1.0 / math.sqrt(head_dim)
    return Batch(name=name, num_q_heads=num_q_heads, num_kv_heads=num_kv_heads, head_dim=head_dim,
                 block_size=block_size, num_blocks=int(num_blocks), scale=float(scale), ctx_lens=ctx,
                 cu_q_lens=np.array(cu, dtype=np.int32), q_positions=q_positions, block_tables=bt,
                 q=q, k_new=k_new, v_new=v_new, used_blocks=used, k_used=k_used, v_used=v_used,
                 kinds=[r.kind for r in requests], seed=seed)


# ---------------------------------------------------------------------------
# The five workloads.  Each is a function of its seed only.
# ---------------------------------------------------------------------------

def _decode(h: int) -> RequestSpec:
    """A decode step: ``h`` cached tokens plus one new token at position ``h``."""
    return RequestSpec(ctx=h + 1, q_positions=np.array([h], np.int32), kind="decode")


def _new_turn(h: int, n: int) -> RequestSpec:
    """A new conversation turn: ``h`` cached tokens plus ``n`` new tokens at ``[h, h+n)``."""
    kind = "prefill" if h == 0 else "new_turn"
    return RequestSpec(ctx=h + n, q_positions=np.arange(h, h + n, dtype=np.int32), kind=kind)


def _recompute(c: int, e: int, n: int) -> RequestSpec:
    """Partial eviction: the leading ``e`` of ``c`` history tokens were dropped and are
    recomputed as query tokens at ``[0, e)`` next to ``n`` new tokens at ``[c, c+n)``."""
    pos = np.concatenate([np.arange(0, e), np.arange(c, c + n)]).astype(np.int32)
    return RequestSpec(ctx=c + n, q_positions=pos, kind="recompute")


def tiny_mixed(seed: int = 1) -> Batch:
    """3 requests, 4 MHA heads, head_dim 64, block 16, pool of 64 blocks.

    A: 40 cached + 8 new; B: 0 cached + 5 new (pure prefill); C: 100 cached + 1 new (decode).
    """
    reqs = [_new_turn(40, 8), _new_turn(0, 5), _decode(100)]
    return build_batch("tiny_mixed", reqs, num_q_heads=4, num_kv_heads=4, head_dim=64,
                       num_blocks=64, seed=seed)


def llama13b_mixed(seed: int = 2) -> Batch:
    """Llama-2-13B attention shape (40 MHA heads, head_dim 128), 32 conversations with
    history ~U[200,2000]; 24 decode, 8 new turns of ~U[50,400] tokens; 60,000-block pool."""
    g = np.random.Generator(np.random.PCG64(np.random.SeedSequence([seed, 101])))
    h = g.integers(200, 2001, size=32)
    turn = np.zeros(32, bool)
    turn[g.permutation(32)[:8]] = True
    n = g.integers(50, 401, size=32)
    reqs = [_new_turn(int(h[i]), int(n[i])) if turn[i] else _decode(int(h[i])) for i in range(32)]
    return build_batch("llama13b_mixed", reqs, num_q_heads=40, num_kv_heads=40, head_dim=128,
                       num_blocks=60000, seed=seed)


def decode_lognormal(seed: int = 3, num_reqs: int = 256) -> Batch:
    """Decode only: 256 requests x 1 token, 40 MHA heads, head_dim 128, context lengths
    round(LogNormal(ln 1500, 0.6)) clipped to [16, 8192]; pool = 1.25 x blocks needed."""
    g = np.random.Generator(np.random.PCG64(np.random.SeedSequence([seed, 103])))
    ctx = np.clip(np.rint(g.lognormal(math.log(1500.0), 0.6, size=num_reqs)), 16, 8192).astype(int)
    reqs = [_decode(int(c) - 1) for c in ctx]
    return build_batch("decode_lognormal", reqs, num_q_heads=40, num_kv_heads=40, head_dim=128,
                       pool_factor=1.25, seed=seed)


def llama70b_gqa(seed: int = 4) -> Batch:
    """Llama-2-70B attention shape (64 query heads, 8 KV heads, head_dim 128), 64
    conversations with history ~U[500,4096]; 48 decode + 16 new turns of ~U[100,800]."""
    g = np.random.Generator(np.random.PCG64(np.random.SeedSequence([seed, 104])))
    h = g.integers(500, 4097, size=64)
    turn = np.zeros(64, bool)
    turn[g.permutation(64)[:16]] = True
    n = g.integers(100, 801, size=64)
    reqs = [_new_turn(int(h[i]), int(n[i])) if turn[i] else _decode(int(h[i])) for i in range(64)]
    return build_batch("llama70b_gqa", reqs, num_q_heads=64, num_kv_heads=8, head_dim=128,
                       pool_factor=1.25, seed=seed)


def long_skewed_evict(seed: int = 5) -> Batch:
    """8 requests, 40 MHA heads, head_dim 128: r0 has 65,536 cached tokens + 1 decode token;
    r1..r7 have histories ~U[512,8192]; in r1..r3 the leading ~U[64,1024] tokens were evicted
    and are recomputed at [0,e) next to ~U[20,200] new-turn tokens; r4..r7 decode."""
    g = np.random.Generator(np.random.PCG64(np.random.SeedSequence([seed, 105])))
    c = g.integers(512, 8193, size=7)
    e = g.integers(64, 1025, size=3)
    n = g.integers(20, 201, size=3)
    reqs = [_decode(65536)]
    for i in range(3):
        reqs.append(_recompute(int(c[i]), int(min(e[i], c[i])), int(n[i])))
    for i in range(3, 7):
        reqs.append(_decode(int(c[i])))
    return build_batch("long_skewed_evict", reqs, num_q_heads=40, num_kv_heads=40, head_dim=128,
                       pool_factor=1.25, seed=seed)


def decode_lognormal_small(seed: int = 3) -> Batch:
    """The decode-only workload cut to 64 requests (about 3 GB of pool): a
    profiling-size case whose KV still far exceeds L2."""
    b = decode_lognormal(seed=seed, num_reqs=64)
    b.name = "decode_lognormal_small"
    return b


WORKLOADS = {
    "tiny_mixed": tiny_mixed,
    "llama13b_mixed": llama13b_mixed,
    "decode_lognormal": decode_lognormal,
    "llama70b_gqa": llama70b_gqa,
    "long_skewed_evict": long_skewed_evict,
    "decode_lognormal_small": decode_lognormal_small,
}


def random_small(seed: int, *, num_q_heads: int = 4, num_kv_heads: int = 2, head_dim: int = 64,
                 num_reqs: int = 5, max_ctx: int = 300, max_q: int = 40) -> Batch:
    """A random small unified batch mixing decode, new-turn, prefill and recompute requests."""
    g = np.random.Generator(np.random.PCG64(np.random.SeedSequence([seed, 999])))
    reqs = []
    for _ in range(num_reqs):
        kind = g.integers(0, 4)
        if kind == 0:
            reqs.append(_decode(int(g.integers(0, max_ctx))))
        elif kind == 1:
            reqs.append(_new_turn(0, int(g.integers(1, max_q + 1))))
        elif kind == 2:
            reqs.append(_new_turn(int(g.integers(1, max_ctx)), int(g.integers(1, max_q + 1))))
        else:
            c = int(g.integers(2, max_ctx))
            e = int(g.integers(1, c))
            reqs.append(_recompute(c, e, int(g.integers(0, max_q + 1))))
    return build_batch(f"random_small_{seed}", reqs, num_q_heads=num_q_heads, num_kv_heads=num_kv_heads,
                       head_dim=head_dim, pool_factor=1.5, seed=seed)


def decode_small(seed: int, *, num_q_heads: int = 4, num_kv_heads: int = 4, head_dim: int = 128,
                 num_reqs: int = 6, max_ctx: int = 3000, tokens: int = 1) -> Batch:
    """A decode-regime batch: every request has ``tokens`` new tokens (tokens * G <= 4 query
    rows per KV head) after a history of ~U[0, max_ctx) cached tokens; one request has the
    full max_ctx so that its keys are split over several items."""
    g = np.random.Generator(np.random.PCG64(np.random.SeedSequence([seed, 555])))
    hist = [int(max_ctx)] + [int(x) for x in g.integers(0, max_ctx, size=num_reqs - 1)]
    reqs = [_decode(h) if tokens == 1 else _new_turn(h, tokens) for h in hist]
    return build_batch(f"decode_small_{seed}", reqs, num_q_heads=num_q_heads, num_kv_heads=num_kv_heads,
                       head_dim=head_dim, pool_factor=1.5, seed=seed)


# ---------------------------------------------------------------------------
# Device copies (input marshalling only).
# ---------------------------------------------------------------------------

def bf16_tensor(bits: np.ndarray, device):
    """A torch bfloat16 tensor holding the given bf16 bit patterns."""
    import torch
    return torch.from_numpy(np.ascontiguousarray(bits).view(np.int16)).to(device).view(torch.bfloat16)


def upload(batch: Batch, device="cuda") -> dict:
    """Device tensors of a batch's per-step inputs: q, k_new, v_new (bf16) and the int32 metadata."""
    import torch
    i32 = lambda a: torch.from_numpy(np.ascontiguousarray(a, dtype=np.int32)).to(device)
    return {
        "q": bf16_tensor(batch.q, device),
        "k_new": bf16_tensor(batch.k_new, device),
        "v_new": bf16_tensor(batch.v_new, device),
        "block_tables": i32(batch.block_tables),
        "ctx_lens": i32(batch.ctx_lens),
        "cu_q_lens": i32(batch.cu_q_lens),
        "q_positions": i32(batch.q_positions),
    }


def fp8_codes(shape, seed: int) -> np.ndarray:
    """Random E4M3 code bytes for synthetic FP8 pool contents: a random sign, exponent
    field uniform in [8, 14] and mantissa field uniform in [0, 7], so magnitudes are
    log-uniform over [2, 240] and no code is NaN (only the bit layout is used here)."""
    g = np.random.Generator(np.random.PCG64(np.random.SeedSequence([seed, 808])))
    f = g.integers(0, 2 * 7 * 8, size=shape, dtype=np.uint8)   # (sign, exponent - 8, mantissa) in one draw
    return ((f // 56) << 7) | ((8 + (f % 56) // 8) << 3) | (f % 8)


FP8_DISTINCT_BLOCKS = 1024


def fp8_pool_arrays(batch: Batch):
    """FP8 pool contents [NB, Hkv, B, D] uint8 for a batch: zero codes outside the used
    blocks; used block i holds row i % FP8_DISTINCT_BLOCKS of a table of random codes
    (fp8_codes), so full-size pools are generated in seconds."""
    shape = (batch.num_blocks, batch.num_kv_heads, 16, batch.head_dim)
    kp, vp = np.zeros(shape, np.uint8), np.zeros(shape, np.uint8)
    u = batch.used_blocks.size
    if u:
        n = (min(u, FP8_DISTINCT_BLOCKS),) + shape[1:]
        pick = np.arange(u) % n[0]
        kp[batch.used_blocks] = fp8_codes(n, batch.seed * 2 + 1)[pick]
        vp[batch.used_blocks] = fp8_codes(n, batch.seed * 2 + 2)[pick]
    return kp, vp


def fill_pool_fp8(batch: Batch, k_storage, v_storage):
    """Write fp8_pool_arrays(batch) into device uint8 storage (used blocks only; zeros elsewhere)."""
    import torch
    k_storage.zero_()
    v_storage.zero_()
    if batch.used_blocks.size:
        kp, vp = fp8_pool_arrays(batch)
        idx = torch.from_numpy(batch.used_blocks.astype(np.int64)).to(k_storage.device)
        k_storage[idx] = torch.from_numpy(kp[batch.used_blocks]).to(k_storage.device)
        v_storage[idx] = torch.from_numpy(vp[batch.used_blocks]).to(v_storage.device)


def fill_pool(batch: Batch, k_storage, v_storage):
    """Write the batch's initial pool contents (used blocks; zeros elsewhere) into device storage."""
    import torch
    k_storage.zero_()
    v_storage.zero_()
    if batch.used_blocks.size:
        idx = torch.from_numpy(batch.used_blocks.astype(np.int64)).to(k_storage.device)
        k_storage[idx] = bf16_tensor(batch.k_used, k_storage.device)
        v_storage[idx] = bf16_tensor(batch.v_used, v_storage.device)
