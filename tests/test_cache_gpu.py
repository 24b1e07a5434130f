"""The two-tier block manager driving the real pool: each step runs the planned
swap-outs and swap-ins with the swap kernels, then appends the step's tokens
(recomputed prefix and new tokens) with the append kernel.  The CPU oracle
runs the same swaps and appends on its own copy of the pool and of the host
buffer: after every step the whole GPU pool and host buffer must equal the
oracle's, bit for bit, and every requested conversation's history, read back
through its block table, must equal the K/V it was given."""
import numpy as np
import pytest
import torch

import oracle
from paged_kv_attention_25_gb300 import build as pkv_build
from paged_kv_attention_25_gb300 import pkv

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module", autouse=True)
def built():
    pkv_build.build()
    oracle.build()


def bits(t: torch.Tensor) -> np.ndarray:
    return t.contiguous().view(torch.int16).cpu().numpy().view(np.uint16)


@pytest.mark.parametrize("seed,gpu_blocks,cpu_blocks", [(0, 24, 16), (1, 20, 0)])
def test_block_manager_keeps_pool_contents_exact(seed, gpu_blocks, cpu_blocks):
    Hkv, D, max_blocks = 2, 64, 8
    rng = np.random.default_rng(seed)
    pool = pkv.Pool(gpu_blocks, Hkv, D)
    cache = pkv.Cache(gpu_blocks, cpu_blocks, 8.0)
    host = torch.zeros((max(cpu_blocks, 1), 2, Hkv, 16, D), dtype=torch.bfloat16).pin_memory()
    kv = {}   # conversation -> [tokens, 2, Hkv, D] bf16: the K/V of every token it has seen
    kp = np.zeros((gpu_blocks, Hkv, 16, D), np.uint16)       # the oracle's pool and host buffer
    vp = np.zeros_like(kp)
    host_ref = np.zeros((max(cpu_blocks, 1), 2, Hkv, 16, D), np.uint16)
    swaps = recomputes = 0
    for step in range(60):
        convs = [int(x) for x in rng.choice(8, size=int(rng.integers(1, 3)), replace=False)]
        new = [int(min(rng.integers(1, 30), max_blocks * 16 - (kv[c].shape[0] if c in kv else 0))) for c in convs]
        try:
            r = cache.step(convs, new, max_blocks)
        except pkv.PkvError:
            continue
        for g, s in r["swap_out"]:
            pkv.pkv_swap_out(pool, [int(g)], host[int(s):int(s) + 1])
            host_ref[int(s):int(s) + 1] = oracle.swap_out(kp, vp, np.array([g], np.int32))
        for s, g in r["swap_in"]:
            pkv.pkv_swap_in(pool, [int(g)], host[int(s):int(s) + 1])
            oracle.swap_in(kp, vp, np.array([g], np.int32), host_ref[int(s):int(s) + 1])
        swaps += len(r["swap_out"]) + len(r["swap_in"])
        # the step's tokens: recomputed prefix [0, rec) with its original K/V, then new tokens
        pos, knew, vnew, cu = [], [], [], [0]
        for k, c in enumerate(convs):
            old = kv[c].shape[0] if c in kv else 0
            fresh = torch.randn((new[k], 2, Hkv, D)).to(torch.bfloat16)
            kv[c] = torch.cat([kv[c], fresh]) if c in kv else fresh
            rec = int(r["recompute"][k])
            recomputes += rec > 0
            p = list(range(rec)) + list(range(old, old + new[k]))
            pos += p
            knew.append(kv[c][p, 0])
            vnew.append(kv[c][p, 1])
            cu.append(cu[-1] + len(p))
        if pos:
            kn, vn = torch.cat(knew).contiguous(), torch.cat(vnew).contiguous()
            pkv.pkv_append(pool, torch.from_numpy(r["block_tables"]).cuda(), torch.tensor(cu, dtype=torch.int32).cuda(),
                           torch.tensor(pos, dtype=torch.int32).cuda(), kn.cuda(), vn.cuda())
            oracle.append(kp, vp, r["block_tables"], np.array(cu, np.int32), np.array(pos, np.int32), bits(kn),
                          bits(vn))
        torch.cuda.synchronize()
        assert pkv.pkv_check_device_errors(pool) == 0
        assert np.array_equal(bits(pool.k), kp) and np.array_equal(bits(pool.v), vp), f"step {step}: pool vs oracle"
        assert np.array_equal(bits(host), host_ref), f"step {step}: host buffer vs oracle"
        pk, pv = pool.k.cpu(), pool.v.cpu()
        for k, c in enumerate(convs):
            n = int(r["ctx_lens"][k])
            assert n == kv[c].shape[0]
            tbl = r["block_tables"][k]
            got_k = torch.stack([pk[int(tbl[p // 16]), :, p % 16] for p in range(n)])
            got_v = torch.stack([pv[int(tbl[p // 16]), :, p % 16] for p in range(n)])
            assert torch.equal(got_k.view(torch.int16), kv[c][:, 0].contiguous().view(torch.int16)), f"step {step} conv {c}"
            assert torch.equal(got_v.view(torch.int16), kv[c][:, 1].contiguous().view(torch.int16)), f"step {step} conv {c}"
    assert recomputes > 0 and (cpu_blocks == 0 or swaps > 0)
    pool.close()
