"""Host-side block pool / block table / copy-on-write bookkeeping against the block
maps the pages print (tests/golden/block_maps.json)."""
import json
from pathlib import Path

import pytest

from paged_kv_cache_90_gb300.block_manager import (BlockAllocator, BlockManager, PoolExhausted,
                                                   blocks_needed, validate_cow_pairs)

G = json.loads((Path(__file__).parent / "golden" / "block_maps.json").read_text())


def _mgr(nb, bs, first):
    order = list(first) + [b for b in range(nb) if b not in first]
    return BlockManager(BlockAllocator(nb, bs, order))


def test_table_example_slots():
    g = G["table_example"]
    bs = g["block_size"]
    m = _mgr(16, bs, g["block_table"])
    slots = m.add_sequence(0, g["num_tokens"])
    assert m.seqs[0].blocks == g["block_table"]
    for lb, (lo, hi) in enumerate(g["token_ranges"]):
        for t in range(lo, hi + 1):
            assert slots[t] == g["block_table"][lb] * bs + t % bs
    m.check_structure()


def test_teaching_map_growth_and_free():
    g = G["teaching_map"]
    bs = g["block_size"]
    m = _mgr(16, bs, [7, 2, 9, 4])
    m.add_sequence("A", g["A_len"])
    m.add_sequence("B", g["B_len"])
    assert m.seqs["A"].blocks == g["A_table"]
    assert m.seqs["B"].blocks == g["B_table"]
    reserved = sum(len(s.blocks) * bs for s in m.seqs.values())
    used = sum(s.length for s in m.seqs.values())
    assert (used, reserved, reserved - used) == (g["slots_used"], g["slots_reserved"],
                                                 g["internal_remainder"])
    for _ in range(g["A_grown_len"] - g["A_len"]):
        m.append_token("A")
    assert m.seqs["A"].blocks == g["A_grown_table"]
    m.check_structure()
    free_before = m.alloc.num_free
    m.free_sequence("B")
    assert m.alloc.num_free == free_before + 1
    for b in g["freed_when_B_ends"]:
        assert m.alloc.is_free(b)
    m.check_structure()


def test_on_demand_demo():
    g = G["on_demand_demo"]
    bs = g["block_size"]
    m = BlockManager(BlockAllocator(8, bs))
    m.add_sequence(0, g["prompt_tokens"])
    assert len(m.seqs[0].blocks) == g["prompt_blocks"] == blocks_needed(g["prompt_tokens"], bs)
    while m.seqs[0].length < 32:
        m.append_token(0)
    assert len(m.seqs[0].blocks) == g["at_32_blocks"]
    m.append_token(0)
    assert len(m.seqs[0].blocks) == g["at_33_blocks"] == blocks_needed(33, bs)
    assert m.seqs[0].blocks == g["table_after_33"]
    m.free_sequence(0)
    assert m.alloc.num_free == 8


def test_internal_fragmentation_examples():
    g = G["internal_fragmentation"]
    m = BlockManager(BlockAllocator(4, g["block_size"]))
    m.add_sequence(0, g["num_tokens"])
    assert len(m.seqs[0].blocks) == g["blocks"]
    assert m.unused_slots(0) == g["empty_slots"]
    g = G["five_positions"]
    m = _mgr(8, g["block_size"], g["logical_to_physical"])
    m.add_sequence(0, g["num_tokens"])
    assert len(m.seqs[0].blocks) * g["block_size"] == g["slots"]
    assert m.seqs[0].blocks == g["logical_to_physical"]


def test_shared_prompt_refcounts_and_copy_on_write():
    g = G["shared_prompt"]
    bs = g["block_size"]
    m = BlockManager(BlockAllocator(32, bs))
    m.add_sequence("P", g["prompt_tokens"])
    prompt = list(m.seqs["P"].blocks)
    assert len(prompt) == g["prompt_blocks"]
    for name, extra in g["private_blocks"].items():
        m.fork("P", name)
        for _ in range(extra * bs):
            _, pair = m.append_token(name)
            assert pair is None          # the prompt ends on a block boundary
    m.free_sequence("P")
    for b in prompt:
        assert m.alloc.refcount[b] == len(g["private_blocks"])
    for name, extra in g["private_blocks"].items():
        assert m.seqs[name].blocks[:len(prompt)] == prompt
        assert len(m.seqs[name].blocks) == len(prompt) + extra
    m.check_structure()


def test_copy_on_write_mid_block():
    """Four samples share a partly filled block: the first three writers get private
    copies, the last writes in place, and every pair's source is the shared block."""
    m = BlockManager(BlockAllocator(16, 4))
    m.add_sequence(0, 6)
    for j in (1, 2, 3):
        m.fork(0, j)
    shared = m.seqs[0].blocks[1]
    assert m.alloc.refcount[shared] == 4
    pairs = []
    for j in range(4):
        slot, pair = m.append_token(j)
        if pair:
            pairs.append(pair)
        assert slot == m.seqs[j].blocks[1] * 4 + 2
    assert len(pairs) == 3 and all(p[0] == shared for p in pairs)
    assert m.seqs[3].blocks[1] == shared and m.alloc.refcount[shared] == 1
    validate_cow_pairs(pairs, 16)
    m.check_structure()


def test_structural_check_catches_planted_faults():
    m = BlockManager(BlockAllocator(8, 4))
    m.add_sequence(0, 5)
    m.check_structure()
    m.alloc.refcount[m.seqs[0].blocks[0]] += 1          # refcount that no table explains
    with pytest.raises(AssertionError):
        m.check_structure()
    m = BlockManager(BlockAllocator(8, 4))
    m.add_sequence(0, 5)
    m.seqs[0].length = 9                                # table no longer covers the tokens
    with pytest.raises(AssertionError):
        m.check_structure()
    m = BlockManager(BlockAllocator(8, 4))
    m.add_sequence(0, 5)
    m.alloc._free.append(m.seqs[0].blocks[0])           # dangling: referenced and free
    with pytest.raises(AssertionError):
        m.check_structure()


def test_pool_exhaustion_and_bad_pairs():
    m = BlockManager(BlockAllocator(2, 4))
    m.add_sequence(0, 8)
    with pytest.raises(PoolExhausted):
        m.append_token(0)
    with pytest.raises(ValueError):
        validate_cow_pairs([(0, 1), (2, 1)], 4)
    with pytest.raises(ValueError):
        validate_cow_pairs([(0, 1), (1, 2)], 4)
    with pytest.raises(ValueError):
        validate_cow_pairs([(0, 9)], 4)


def test_release_outside_window():
    """40 tokens at 16 per block with a window of 16: positions 24..39 are attended,
    so block 0 (positions 0..15) is released and blocks 1 and 2 stay; releasing is
    idempotent and the block returns to the free list."""
    from paged_kv_cache_90_gb300.block_manager import RELEASED
    mgr = BlockManager(BlockAllocator(8, 16, list(range(8))))
    mgr.add_sequence("a", 40)
    blocks = list(mgr.seqs["a"].blocks)
    free0 = mgr.alloc.num_free
    assert mgr.release_outside_window("a", 16) == [blocks[0]]
    assert mgr.seqs["a"].blocks == [RELEASED] + blocks[1:]
    assert mgr.release_outside_window("a", 16) == []
    assert mgr.alloc.num_free == free0 + 1
    mgr.check_structure()
    with pytest.raises(IndexError):
        mgr.seqs["a"].slot(3, 16)
    assert mgr.seqs["a"].slot(24, 16) == blocks[1] * 16 + 8
    # the released block is handed out again; the structure stays consistent
    mgr.add_sequence("b", 16 * 6)
    mgr.check_structure()
    # a window of one token keeps only the block holding the last position
    mgr.release_outside_window("a", 1)
    assert mgr.seqs["a"].blocks[:2] == [RELEASED, RELEASED]
    mgr.check_structure()
    mgr.free_sequence("a")
    mgr.check_structure()


# ---- prefix caching --------------------------------------------------------------

def _kv_of(tokens, pos):
    """Stand-in for a layer's key at a position: a function of the prefix it sees
    (the token and everything before it), as a model's keys are."""
    return hash((tuple(tokens[:pos + 1]),)) & 0xFFFFFFFF


def _pool_with_cache(num_blocks=64, bs=16):
    from paged_kv_cache_90_gb300.block_manager import PrefixCache
    mgr = BlockManager(BlockAllocator(num_blocks, bs, free_order=list(reversed(range(num_blocks)))))
    return mgr, PrefixCache(mgr)


def test_prefix_cache_shares_full_blocks_of_a_common_prefix():
    """Two prompts with a common 32-token prefix at 16 tokens per block: the second
    shares both full blocks and computes only its own 9 tokens; the tables agree on
    the shared blocks and every slot the second prompt reads holds its own keys."""
    mgr, pc = _pool_with_cache()
    a = list(range(100, 140))                       # 40 tokens: blocks 0, 1 full, 2 partial
    b = a[:32] + list(range(500, 509))              # 41 tokens
    pool = {}
    slots, cached = pc.add_prompt("a", a)
    assert cached == 0 and len(slots) == 40
    for pos, sl in enumerate(slots):
        pool[sl] = _kv_of(a, pos)
    slots, cached = pc.add_prompt("b", b)
    assert cached == 32 and len(slots) == 9
    for i, sl in enumerate(slots):
        pool[sl] = _kv_of(b, 32 + i)
    assert mgr.seqs["b"].blocks[:2] == mgr.seqs["a"].blocks[:2]
    assert mgr.seqs["b"].blocks[2] != mgr.seqs["a"].blocks[2]
    for pos in range(len(b)):                       # what attention gathers through b's table
        assert pool[mgr.seqs["b"].slot(pos, 16)] == _kv_of(b, pos)
    mgr.check_structure(held=pc.held())


def test_prefix_cache_identity_is_chained_and_conditioned():
    mgr, pc = _pool_with_cache()
    a = list(range(48))
    pc.add_prompt("a", a)
    assert pc.add_prompt("lora", a + [7], extra=("adapter", 3))[1] == 0   # other conditions
    c = list(a)
    c[3] = 999                                                            # block 0 differs
    assert pc.add_prompt("c", c + [7])[1] == 0                            # so no later block matches
    d = list(a)
    d[20] = 999                                                           # block 1 differs
    assert pc.add_prompt("d", d + [7])[1] == 16
    assert pc.add_prompt("e", a[:40])[1] == 32                            # partial last block: never shared
    assert pc.add_prompt("f", a)[1] == 32                                 # cached whole: the last block is recomputed
    assert mgr.seqs["f"].blocks[2] != mgr.seqs["a"].blocks[2]
    mgr.check_structure(held=pc.held())


def test_prefix_cache_outlives_sequences_until_evicted():
    mgr, pc = _pool_with_cache(num_blocks=8)
    a = list(range(40))
    pc.add_prompt("a", a)                            # 3 blocks, 2 identified
    mgr.free_sequence("a")
    assert mgr.alloc.num_free == 6                   # the cache still holds the 2 full blocks
    mgr.check_structure(held=pc.held())
    assert pc.add_prompt("b", a)[1] == 32            # a later request finds them
    assert pc.evict(10) == 0                         # b holds them: nothing to drop
    mgr.free_sequence("b")
    assert pc.evict(1) == 1 and mgr.alloc.num_free == 7   # least recently used first
    assert pc.evict(10) == 1 and mgr.alloc.num_free == 8
    assert pc.held() == []
    mgr.check_structure()
    assert pc.add_prompt("c", a)[1] == 0
