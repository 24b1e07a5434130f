"""Host-only tests of the two-tier block manager (pkv_cache_*): hand-built
scenarios that fix the eviction order, and random traces checked by a content
model that executes the returned swap lists and requires every retained block
to hold its own conversation's data."""
import numpy as np
import pytest

from paged_kv_attention_25_gb300 import build as pkv_build
from paged_kv_attention_25_gb300 import pkv


@pytest.fixture(scope="module", autouse=True)
def lib():
    pkv_build.build()
    return pkv.load_library()


def test_new_conversations_get_fresh_blocks():
    c = pkv.Cache(16, 4)
    r = c.step([5, 9], [40, 16], 8)
    assert list(r["ctx_lens"]) == [40, 16] and list(r["recompute"]) == [0, 0]
    assert (r["block_tables"][0, :3] >= 0).all() and (r["block_tables"][0, 3:] == -1).all()
    assert (r["block_tables"][1, :1] >= 0).all() and (r["block_tables"][1, 1:] == -1).all()
    assert len(set(r["block_tables"][r["block_tables"] >= 0].tolist())) == 4
    assert len(r["swap_out"]) == 0 and len(r["swap_in"]) == 0
    # growing in place: 40 -> 48 tokens fills the last block; 48 -> 50 needs a fourth
    r2 = c.step([5], [8], 8)
    assert list(r2["block_tables"][0, :3]) == list(r["block_tables"][0, :3]) and r2["block_tables"][0, 3] == -1
    assert c.free_blocks() == (12, 4)
    r3 = c.step([5], [2], 8)
    assert list(r3["block_tables"][0, :3]) == list(r["block_tables"][0, :3]) and r3["block_tables"][0, 3] >= 0
    assert c.free_blocks() == (11, 4)


def test_idle_conversation_moves_leading_blocks_to_cpu_and_back():
    # Recompute cost of a full block b (token_cost 0): 256 b + 136.
    c = pkv.Cache(6, 8)
    a = c.step([0], [64], 8)["block_tables"][0, :4]          # A: 4 blocks (step 1)
    b = c.step([1], [32], 8)["block_tables"][0, :2]          # B: 2 blocks (step 2), pool full
    r = c.step([2], [32], 8)                                 # C needs 2 (step 3)
    # first victim: A's block 0 (idle 2 / 136 beats B's idle 1 / 136); then A's
    # leading block is block 1 (2 / 392), so B's block 0 (1 / 136) goes second
    assert [(int(g), int(s)) for g, s in r["swap_out"]] == [(int(a[0]), int(r["swap_out"][0][1])),
                                                            (int(b[0]), int(r["swap_out"][1][1]))]
    # A returns: its CPU block comes back in front, nothing is recomputed
    back = c.step([0], [1], 8)
    assert back["recompute"][0] == 0 and back["ctx_lens"][0] == 65
    assert [int(x) for x in back["swap_in"][:, 0]] == [int(r["swap_out"][0][1])]
    tbl = back["block_tables"][0]
    assert int(tbl[0]) == int(back["swap_in"][0][1]) and list(tbl[1:4]) == list(a[1:4])


def test_without_cpu_tier_leading_blocks_are_recomputed():
    c = pkv.Cache(4, 0)
    c.step([0], [40], 8)                 # 3 blocks (last one partial)
    r = c.step([1], [32], 8)             # needs 2, 1 free: A drops its leading block
    assert len(r["swap_out"]) == 0
    back = c.step([0], [8], 8)           # A needs its 3 blocks again plus room for 48 tokens (3 blocks)
    assert back["recompute"][0] == 16 and back["ctx_lens"][0] == 48
    # B lost its leading block to make room for A, and recomputes it on return
    again = c.step([1], [0], 8)
    assert again["recompute"][0] == 16


def test_longest_idle_conversation_is_evicted_first():
    c = pkv.Cache(6, 8)
    c.step([0], [32], 8)      # A at step 1
    c.step([1], [32], 8)      # B at step 2
    c.step([2], [32], 8)      # C at step 3: pool full
    r = c.step([3], [16], 8)  # one block: A (idle 3) before B (idle 2) before C (idle 1)
    a_tbl = c.step([0], [0], 8)  # A returns: its leading block comes back from the CPU tier
    assert len(r["swap_out"]) == 1 and len(a_tbl["swap_in"]) == 1
    assert a_tbl["swap_in"][0][0] == r["swap_out"][0][1]


def test_cheaper_leading_block_is_evicted_first_at_equal_idle():
    # A and B requested in the same step (equal idle); A's leading GPU block sits at
    # a later position (its first block already went to the CPU tier), so B's
    # position-0 block is the cheaper one to recompute and goes first.
    c = pkv.Cache(5, 8)
    c.step([0, 1], [32, 32], 8)          # A: blocks 0,1; B: blocks 0,1 -> 1 free
    c.step([2], [16], 8)                 # C takes the last free block
    r1 = c.step([3], [16], 8)            # one more: A and B tie on idle and cost -> lower id (A) goes
    assert len(r1["swap_out"]) == 1
    c2 = pkv.Cache(5, 8)
    c2.step([0, 1], [32, 32], 8)
    c2.step([2], [16], 8)
    c2.step([3], [16], 8)                # A's block 0 moved to the CPU tier
    r2 = c2.step([4], [16], 8)           # next victim: B's block 0 (position 0) beats A's block 1 (position 16)
    b_back = c2.step([1], [0], 8)
    assert len(b_back["swap_in"]) == 1 and b_back["swap_in"][0][0] == r2["swap_out"][0][1]


def test_token_cost_weighs_idle_time_against_position():
    # With no fixed cost per token, A's second block (position 16, cost 392) is
    # dearer than another idle conversation's first block (136), so that one
    # goes; with a large fixed cost every block costs about the same and the
    # longest idle conversation (A) loses its second block too.
    def victim(token_cost):
        c = pkv.Cache(5, 8, token_cost)
        c.step([0], [32], 8)             # A (idle longer)
        c.step([1], [16], 8)             # B
        c.step([2], [16], 8)
        c.step([3], [16], 8)             # pool full (2 + 1 + 1 + 1)
        c.step([4], [16], 8)             # evicts A block 0 either way (oldest, position 0)
        c.step([1], [16], 8)             # B requested again: B becomes fresh, A stays idle
        r = c.step([5], [16], 8)
        owner = c.step([0], [0], 8)      # does A get a block back from the CPU tier for position 16?
        return len(owner["swap_in"])
    assert victim(0.0) == 1
    assert victim(1e6) == 2


def test_not_enough_room_is_an_error_and_changes_nothing():
    c = pkv.Cache(4, 4)
    c.step([0], [32], 8)
    before = c.free_blocks()
    with pytest.raises(pkv.PkvError):
        c.step([0, 1], [0, 48], 8)       # A keeps 2 blocks, B wants 3: 5 > 4
    assert c.free_blocks() == before
    r = c.step([1], [48], 8)             # alone it fits after evicting A
    assert len(r["swap_out"]) == 1


def test_bad_arguments_are_rejected():
    c = pkv.Cache(4, 4)
    with pytest.raises(pkv.PkvError):
        c.step([1, 1], [1, 1], 8)
    with pytest.raises(pkv.PkvError):
        c.step([1], [200], 8)            # needs 13 blocks > max_blocks
    with pytest.raises(pkv.PkvError):
        c.step([-1], [1], 8)


@pytest.mark.parametrize("seed,gpu,cpu", [(1, 24, 16), (2, 24, 0), (3, 40, 8), (4, 16, 64)])
def test_random_traces_keep_every_retained_block_intact(seed, gpu, cpu):
    rng = np.random.default_rng(seed)
    c = pkv.Cache(gpu, cpu, float(rng.uniform(0, 64)))
    max_blocks = 8
    length = {}                       # conversation -> tokens the caller believes it has
    gpu_label = {}                    # pool block -> (conv, block index) whose data it holds
    cpu_label = {}                    # host slot -> (conv, block index)
    tables = {}
    for step in range(200):
        conv_ids = rng.choice(12, size=int(rng.integers(1, 4)), replace=False)
        new = [int(rng.integers(0, 24)) for _ in conv_ids]
        new = [min(n, max_blocks * 16 - length.get(int(cv), 0)) for cv, n in zip(conv_ids, new)]
        try:
            r = c.step(conv_ids, new, max_blocks)
        except pkv.PkvError:
            continue
        # execute the swaps in the documented order on the content model
        for g, s in r["swap_out"]:
            assert int(g) in gpu_label, "swap-out of a block that holds nothing"
            conv, idx = gpu_label.pop(int(g))
            assert conv not in set(int(x) for x in conv_ids), "a requested conversation was evicted"
            cpu_label[int(s)] = (conv, idx)   # a slot's earlier block may have been dropped: no copy shows it
        for s, g in r["swap_in"]:
            cpu_label_pair = cpu_label.pop(int(s))
            gpu_label[int(g)] = cpu_label_pair
        for k, cv in enumerate(int(x) for x in conv_ids):
            old = length.get(cv, 0)
            tbl = r["block_tables"][k]
            nblk = -(-int(r["ctx_lens"][k]) // 16)
            assert int(r["ctx_lens"][k]) == old + new[k]
            assert (tbl[:nblk] >= 0).all() and (tbl[:nblk] < gpu).all() and (tbl[nblk:] == -1).all()
            rec = int(r["recompute"][k])
            assert rec == old or rec % 16 == 0, "recompute is a block-aligned prefix"
            assert rec <= old
            for idx in range(nblk):
                g = int(tbl[idx])
                if idx * 16 >= rec and idx * 16 < old:   # retained history: must hold its own data
                    assert gpu_label.get(g) == (cv, idx), f"step {step}: conv {cv} block {idx} lost"
                gpu_label[g] = (cv, idx)               # recomputed / new / retained: now holds this block
            length[cv] = old + new[k]
            tables[cv] = tbl[:nblk].copy()
        # every pool block holds at most one conversation block
        owners = [t for t in gpu_label.values()]
        assert len(owners) == len(set(owners))
        free_gpu, free_cpu = c.free_blocks()
        assert free_gpu <= gpu and free_cpu <= cpu
