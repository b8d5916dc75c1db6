"""Pins for the CPU oracle: values the pages print, closed forms, invariants, and
library routines that the oracle's arithmetic reduces to.  None of these needs a GPU
and none of them reads the oracle's own code back as its expectation."""
import itertools
import json
import math
from pathlib import Path

import numpy as np
import pytest
import torch

import oracle
from paged_kv_cache_90_gb300 import workloads as wl
from paged_kv_cache_90_gb300.block_manager import BlockAllocator, BlockManager

GOLDEN = Path(__file__).parent / "golden"


@pytest.fixture(scope="module", autouse=True)
def _build_oracle():
    oracle.build()


def _materialize(w, step=0):
    """Caches after the step's copy-on-write pairs and new-token writes (the state
    the decode of that step reads)."""
    st = w.steps[step]
    kc, vc = w.key_cache.clone(), w.value_cache.clone()
    if st.cow_pairs.numel():
        oracle.copy_blocks(kc, st.cow_pairs)
        oracle.copy_blocks(vc, st.cow_pairs)
    if st.slot_mapping.numel():
        oracle.reshape_and_cache(st.new_key, st.new_value, kc, vc, st.slot_mapping,
                                 w.k_scale, w.v_scale)
    return kc, vc


def _decode(w, step=0, kc=None, vc=None):
    st = w.steps[step]
    if kc is None:
        kc, vc = _materialize(w, step)
    return oracle.paged_attention_decode(st.query, kc, vc, st.block_tables, st.context_lens,
                                         w.scale, w.k_scale, w.v_scale)


# --- the scalar worked example ----------------------------------------------------

def test_scalar_example_printed_layouts():
    g = json.loads((GOLDEN / "scalar_example.json").read_text())
    for layout in g["layouts"]:
        w = wl.scalar_example(physical=layout, num_blocks=8)
        out = _decode(w)
        assert out.shape == (1, 1, 1)
        assert abs(float(out[0, 0, 0]) - g["expected_output"]) <= 4 * np.finfo(np.float64).eps * 3


@pytest.mark.parametrize("head_dim", [1, 64])
def test_scalar_example_every_layout(head_dim):
    """Output 3 for every placement of the two logical blocks in a pool of 6; a head
    padded with zeros to 64 dims leaves column 0 at 3 and the rest at 0."""
    for a, b in itertools.permutations(range(6), 2):
        w = wl.scalar_example(physical=(a, b), num_blocks=6, head_dim=head_dim)
        out = _decode(w)[0, 0]
        assert abs(float(out[0]) - 3.0) <= 1e-15
        assert torch.all(out[1:] == 0)


# --- closed forms -----------------------------------------------------------------

def _small(seed, lengths, hq=4, hk=2, d=16, bs=4, kv="bf16", q="bf16", poison=False):
    return wl.variable_length_decode("t", seed, lengths, hq, hk, d, bs, kv, q_dtype=q,
                                     poison=poison)


def _gather(cache, table, k, L, bs):
    """Contiguous [L, D] rows of KV head k for one sequence, by torch indexing."""
    n = -(-L // bs)
    blocks = cache[table[:n].long()]            # [n, Hk, bs, D]
    return blocks[:, k].reshape(n * bs, -1)[:L]


def test_single_token_returns_its_value():
    """L = 1: the one weight is exactly 1, so the output is V[0] exactly."""
    w = _small(11, [1, 1, 1], kv="bf16")
    kc, vc = _materialize(w)
    out = _decode(w, kc=kc, vc=vc)
    st = w.steps[0]
    for s in range(3):
        for h in range(w.num_heads):
            k = h // (w.num_heads // w.num_kv_heads)
            v0 = _gather(vc, st.block_tables[s], k, 1, w.block_size)[0].double()
            assert torch.equal(out[s, h], v0)


def test_equal_keys_give_mean_of_values():
    """All keys equal -> all weights 1/L -> output = mean of the values (the scalar
    example's argument, for any L and any head_dim)."""
    w = _small(12, [7, 33, 50], d=32, kv="f32", q="f32")
    kc, vc = _materialize(w)
    kc[:] = 0.25
    out = _decode(w, kc=kc, vc=vc)
    st = w.steps[0]
    for s in range(3):
        L = int(st.context_lens[s])
        for h in range(w.num_heads):
            k = h // (w.num_heads // w.num_kv_heads)
            mean = _gather(vc, st.block_tables[s], k, L, w.block_size).double().mean(0)
            assert torch.allclose(out[s, h], mean, rtol=0, atol=1e-14)


def test_peaked_scores_select_one_value():
    """One key aligned with the query by a margin Delta over the others: the output is
    within 2 * max|V| * (L-1) e^-Delta of that key's value."""
    d, L, bs = 16, 24, 8
    w = _small(13, [L], hq=1, hk=1, d=d, bs=bs, kv="f32", q="f32")
    st = w.steps[0]
    st.query.zero_()
    st.query[0, 0, 0] = 1.0
    jstar, delta = 17, 40.0
    table = st.block_tables[0]
    kc, vc = _materialize(w)
    for j in range(L):
        blk, off = int(table[j // bs]), j % bs
        kc[blk, 0, off].zero_()
        kc[blk, 0, off, 0] = delta if j == jstar else 0.0
    w.scale = 1.0
    out = _decode(w, kc=kc, vc=vc)[0, 0]
    v = _gather(vc, table, 0, L, bs).double()
    bound = 2 * v.abs().max() * (L - 1) * math.exp(-delta)
    assert torch.max(torch.abs(out - v[jstar])) <= bound + 1e-15


# --- equality with dense attention (a library routine) ------------------------------

@pytest.mark.parametrize("kv,q,hq,hk,d,bs", [
    ("f32", "f32", 4, 4, 64, 16),
    ("bf16", "bf16", 8, 2, 128, 16),
    ("bf16", "bf16", 4, 1, 64, 8),
    ("bf16", "f32", 6, 2, 64, 32),
    ("e4m3", "bf16", 8, 2, 128, 16),
    ("f32", "f32", 3, 3, 16, 4),
])
def test_equals_dense_sdpa(kv, q, hq, hk, d, bs):
    """Paged attention equals contiguous attention over the gathered context:
    torch's scaled_dot_product_attention in float64, K/V heads repeated for the query
    groups, against the oracle."""
    lens = [1, 5, bs, bs + 1, 3 * bs - 1, 70]
    w = _small(20 + d + bs, lens, hq=hq, hk=hk, d=d, bs=bs, kv=kv, q=q, poison=True)
    kc, vc = _materialize(w)
    out = _decode(w, kc=kc, vc=vc)
    st = w.steps[0]
    g = hq // hk
    for s, L in enumerate(st.context_lens.tolist()):
        ks = torch.stack([_gather(kc, st.block_tables[s], k, L, bs) for k in range(hk)])
        vs = torch.stack([_gather(vc, st.block_tables[s], k, L, bs) for k in range(hk)])
        ks = ks.double() * w.k_scale
        vs = vs.double() * w.v_scale
        ks = ks.repeat_interleave(g, dim=0)[None]      # [1, Hq, L, D]
        vs = vs.repeat_interleave(g, dim=0)[None]
        qs = st.query[s].double()[None, :, None, :]    # [1, Hq, 1, D]
        ref = torch.nn.functional.scaled_dot_product_attention(qs, ks, vs, scale=w.scale)
        assert torch.allclose(out[s], ref[0, :, 0], rtol=0, atol=1e-12), (s, L)


# --- invariants ---------------------------------------------------------------------

def test_physical_permutation_invariance():
    """Moving blocks to other physical ids (and renumbering the tables) leaves the
    output bit-identical."""
    w = _small(31, [9, 40, 65, 3], kv="bf16", poison=True)
    k0, v0 = _materialize(w)
    base = _decode(w, kc=k0, vc=v0)
    g = torch.Generator().manual_seed(99)
    perm = torch.randperm(w.num_blocks, generator=g)
    kc = torch.empty_like(k0)
    vc = torch.empty_like(v0)
    kc[perm] = k0
    vc[perm] = v0
    st = w.steps[0]
    bt = st.block_tables.clone()
    used = bt >= 0
    bt[used] = perm[bt[used].long()].to(torch.int32)
    moved = oracle.paged_attention_decode(st.query, kc, vc, bt, st.context_lens, w.scale)
    assert torch.equal(base, moved)


def test_shared_prefix_equals_private_copies():
    """Tables that share physical blocks give the same output as tables whose blocks
    were first copied into private blocks."""
    w = wl.shared_prefix_cow(seed=4, num_groups=3, group_size=4, prefix_blocks=4,
                             suffix_range=(5, 40), poison=True)
    kc, vc = w.key_cache.clone(), w.value_cache.clone()
    shared = oracle.run_workload_step(w, 0, kc, vc)
    st = w.steps[0]
    s = st.block_tables.shape[0]
    nblk = [-(-int(L) // w.block_size) for L in st.context_lens]
    total = sum(nblk)
    kp = torch.full((total,) + tuple(kc.shape[1:]), float("nan"), dtype=kc.dtype)
    vp = torch.full_like(kp, float("nan"))
    bt = torch.full((s, st.block_tables.shape[1]), -1, dtype=torch.int32)
    nxt = 0
    for i in range(s):
        for j in range(nblk[i]):
            src = int(st.block_tables[i, j])
            kp[nxt], vp[nxt] = kc[src], vc[src]
            bt[i, j] = nxt
            nxt += 1
    private = oracle.paged_attention_decode(st.query, kp, vp, bt, st.context_lens, w.scale)
    assert torch.equal(shared, private)
    # sharing is real: the prefix blocks appear in every table
    first = set(st.block_tables[:, 0].tolist())
    assert len(first) == 1


def test_unused_slots_are_never_read():
    """NaN in unused tail slots, in unreferenced blocks and -1 table padding leave the
    output equal to the unpoisoned run."""
    clean = _small(41, [3, 17, 31, 64], kv="bf16", poison=False)
    dirty = _small(41, [3, 17, 31, 64], kv="bf16", poison=True)
    a, b = _decode(clean), _decode(dirty)
    assert torch.isfinite(b).all()
    assert torch.equal(a, b)
    assert torch.isnan(dirty.key_cache.float()).any()


def test_zero_length_gives_zeros():
    w = _small(42, [4, 9], kv="f32", q="f32")
    st = w.steps[0]
    st.context_lens[0] = 0
    out = _decode(w)
    assert torch.all(out[0] == 0)


def test_invalid_table_entry_is_reported():
    w = _small(43, [9], kv="f32", q="f32")
    w.steps[0].block_tables[0, 1] = w.num_blocks + 5
    with pytest.raises(ValueError):
        _decode(w)


# --- cache write and copy-on-write -------------------------------------------------

def test_cache_write_block_table_example():
    """12 tokens at 4 per block through table [7, 2, 11]: tokens 0-3 land in physical
    block 7, 4-7 in block 2, 8-11 in block 11, in position order."""
    g = json.loads((GOLDEN / "block_maps.json").read_text())["table_example"]
    bs, n, table = g["block_size"], g["num_tokens"], g["block_table"]
    order = table + [b for b in range(16) if b not in table]
    mgr = BlockManager(BlockAllocator(16, bs, order))
    slots = mgr.add_sequence("r", n)
    assert mgr.seqs["r"].blocks == table
    keys = torch.arange(n * 2 * 8, dtype=torch.float32).view(n, 2, 8)
    kc = torch.full((16, 2, bs, 8), -1.0)
    vc = torch.full((16, 2, bs, 8), -1.0)
    oracle.reshape_and_cache(keys, -keys, kc, vc, torch.tensor(slots))
    for lb, (lo, hi) in enumerate(g["token_ranges"]):
        phys = table[lb]
        for t in range(lo, hi + 1):
            assert torch.equal(kc[phys, :, t % bs], keys[t])
            assert torch.equal(vc[phys, :, t % bs], -keys[t])
    untouched = [b for b in range(16) if b not in table]
    assert torch.all(kc[untouched] == -1.0)


def test_cache_write_pytorch_example_round_trip():
    """40 keys at block size 16 from the free list [41, 7, 19, 2, 33]: table
    [41, 7, 19]; reading the pool back through the table returns the keys intact;
    8 unused slots against 2008 for a 2,048-token reservation."""
    g = json.loads((GOLDEN / "block_maps.json").read_text())["pytorch_example"]
    bs, d, nb, n = g["block_size"], g["head_dim"], g["pool_blocks"], g["num_tokens"]
    free = g["free_blocks"] + [b for b in range(nb) if b not in g["free_blocks"]]
    mgr = BlockManager(BlockAllocator(nb, bs, free))
    slots = mgr.add_sequence("req", n)
    table = mgr.seqs["req"].blocks
    assert len(table) == g["blocks_needed"]
    assert table == g["block_table"]
    keys = torch.randn(n, 1, d, generator=torch.Generator().manual_seed(0))
    pool = torch.zeros(nb, 1, bs, d)
    oracle.reshape_and_cache(keys, keys, pool, pool.clone(), torch.tensor(slots))
    gathered = pool[table][:, 0].reshape(-1, d)[:n]
    assert torch.equal(gathered, keys[:, 0]) == g["keys_intact"]
    assert mgr.unused_slots("req") == g["unused_slots_paged"]
    assert g["reservation"] - n == g["unused_slots_reserved"]


def test_cache_write_skips_negative_slots():
    keys = torch.ones(3, 1, 4)
    kc = torch.zeros(4, 1, 2, 4)
    vc = torch.zeros(4, 1, 2, 4)
    oracle.reshape_and_cache(keys, keys, kc, vc, torch.tensor([-1, 5, -7]))
    assert torch.equal(kc.view(8, 4)[5], torch.ones(4))
    assert float(kc.sum()) == 4.0


def test_copy_blocks_is_whole_block_byte_copy():
    cache = torch.randn(6, 2, 4, 8, generator=torch.Generator().manual_seed(1)).to(torch.bfloat16)
    ref = cache.clone()
    oracle.copy_blocks(cache, [(1, 4), (3, 0)])
    assert torch.equal(cache[4].view(torch.int16), ref[1].view(torch.int16))
    assert torch.equal(cache[0].view(torch.int16), ref[3].view(torch.int16))
    for b in (1, 2, 3, 5):
        assert torch.equal(cache[b].view(torch.int16), ref[b].view(torch.int16))


def test_copy_on_write_step_matches_private_write():
    """After the copy pairs and the write, each sample sees the shared prefix plus
    its own new token; the shared block's other holders keep the old contents."""
    w = wl.shared_prefix_cow(seed=5, num_groups=2, group_size=4, prefix_blocks=2,
                             suffix_range=(3, 30))
    st = w.steps[0]
    assert st.cow_pairs.shape == (2 * 3, 2)
    kc, vc = w.key_cache.clone(), w.value_cache.clone()
    oracle.run_workload_step(w, 0, kc, vc)
    for i in range(st.block_tables.shape[0]):
        L = int(st.context_lens[i])
        slot = int(st.slot_mapping[i])
        blk, off = slot // w.block_size, slot % w.block_size
        assert int(st.block_tables[i, (L - 1) // w.block_size]) == blk
        assert torch.equal(kc[blk, :, off].view(torch.int16), st.new_key[i].view(torch.int16))
        # the rest of that block equals the source block it was copied from
        for s_, d_ in st.cow_pairs.tolist():
            if d_ == blk:
                assert torch.equal(kc[blk, :, :off].view(torch.int16),
                                   w.key_cache[s_, :, :off].view(torch.int16))


# --- number formats --------------------------------------------------------------

def test_e4m3_decode_all_codes_vs_torch():
    codes = np.arange(256, dtype=np.uint8)
    mine = oracle.e4m3_decode(codes)
    ref = torch.from_numpy(codes).view(torch.float8_e4m3fn).double().numpy()
    assert np.array_equal(np.isnan(mine), np.isnan(ref))
    ok = ~np.isnan(ref)
    assert np.array_equal(mine[ok], ref[ok])
    assert np.isnan(mine[[0x7F, 0xFF]]).all()
    assert mine[0x7E] == 448.0 and mine[0x01] == 2.0 ** -9


def test_e4m3_encode_vs_torch_in_range():
    """Round-to-nearest-even against torch's float8_e4m3fn cast, for random values
    over the whole range and for every midpoint between neighbouring codes (and one
    binary32 ulp either side of it)."""
    g = torch.Generator().manual_seed(7)
    rnd = (torch.rand(200000, generator=g) * 2 - 1) * torch.exp2(torch.rand(200000, generator=g) * 22 - 13)
    rnd = rnd.clamp(-448, 448)
    mags = oracle.e4m3_decode(np.arange(0x7F, dtype=np.uint8))
    mids = (mags[:-1] + mags[1:]) / 2
    mids32 = torch.tensor(mids, dtype=torch.float32)
    up = torch.nextafter(mids32, torch.tensor(1e9))
    dn = torch.nextafter(mids32, torch.tensor(-1e9))
    x = torch.cat([rnd, mids32, up, dn, -mids32, -up, -dn, torch.tensor([0.0, -0.0, 448.0, -448.0])])
    x = x.clamp(-448, 448)
    mine = oracle.e4m3_encode(x.numpy())
    ref = x.to(torch.float8_e4m3fn).view(torch.uint8).numpy()
    assert np.array_equal(mine, ref)


def test_e4m3_encode_saturates_and_round_trips():
    big = np.array([448.0001, 464.0, 1e6, 3e38, np.inf], dtype=np.float32)
    assert np.all(oracle.e4m3_encode(big) == 0x7E)
    assert np.all(oracle.e4m3_encode(-big) == 0xFE)
    assert oracle.e4m3_encode(np.array([np.nan], dtype=np.float32))[0] == 0x7F
    codes = np.array([c for c in range(256) if c not in (0x7F, 0xFF)], dtype=np.uint8)
    vals = oracle.e4m3_decode(codes).astype(np.float32)
    assert np.array_equal(oracle.e4m3_encode(vals), codes)


def test_bf16_decode_all_patterns_vs_torch():
    bits = np.arange(65536, dtype=np.uint32).astype(np.uint16)
    mine = oracle.bf16_decode(bits)
    ref = torch.from_numpy(bits.view(np.int16)).view(torch.bfloat16).double().numpy()
    assert np.array_equal(np.isnan(mine), np.isnan(ref))
    ok = ~np.isnan(ref)
    assert np.array_equal(mine[ok], ref[ok])


def test_fp8_cache_write_matches_torch_cast():
    """The 8-bit cache write (binary32 division by the per-tensor scale, then e4m3)
    agrees with torch's cast of the same quotient for in-range data."""
    w = _small(51, [5, 9], kv="e4m3", d=64, bs=8)
    st = w.steps[0]
    kc, vc = w.key_cache.clone(), w.value_cache.clone()
    oracle.reshape_and_cache(st.new_key, st.new_value, kc, vc, st.slot_mapping,
                             w.k_scale, w.v_scale)
    for t, slot in enumerate(st.slot_mapping.tolist()):
        blk, off = slot // w.block_size, slot % w.block_size
        qk = (st.new_key[t].float() / w.k_scale).clamp(-448, 448).to(torch.float8_e4m3fn)
        qv = (st.new_value[t].float() / w.v_scale).clamp(-448, 448).to(torch.float8_e4m3fn)
        assert torch.equal(kc[blk, :, off].view(torch.uint8), qk.view(torch.uint8))
        assert torch.equal(vc[blk, :, off].view(torch.uint8), qv.view(torch.uint8))


# --- sliding-window decode ------------------------------------------------------------

def _decode_w(w, window, step=0, kc=None, vc=None, tables=None):
    st = w.steps[step]
    if kc is None:
        kc, vc = _materialize(w, step)
    bt = st.block_tables if tables is None else tables
    return oracle.paged_attention_decode(st.query, kc, vc, bt, st.context_lens, w.scale, w.k_scale,
                                         w.v_scale, sliding_window=window)


def test_window_covering_the_context_is_full_attention():
    """A window at least as long as every context changes nothing, bit for bit."""
    w = _small(41, [1, 7, 33, 64], poison=True)
    kc, vc = _materialize(w)
    full = _decode(w, kc=kc, vc=vc)
    for window in (64, 65, 1000):
        assert torch.equal(_decode_w(w, window, kc=kc, vc=vc), full)
    assert torch.equal(_decode_w(w, 0, kc=kc, vc=vc), full)


def test_window_of_one_returns_the_newest_value():
    """W = 1: only the token just written is attended, so the output is its value
    exactly, whatever the queries and keys."""
    w = _small(42, [1, 6, 17, 40], kv="f32", q="f32", poison=True)
    kc, vc = _materialize(w)
    out = _decode_w(w, 1, kc=kc, vc=vc)
    st = w.steps[0]
    g = 4 // 2
    for s, L in enumerate(st.context_lens.tolist()):
        for h in range(4):
            v = _gather(vc, st.block_tables[s], h // g, L, 4)[L - 1].double()
            assert torch.equal(out[s, h], v)


@pytest.mark.parametrize("bs", [4, 8, 16])
@pytest.mark.parametrize("window", [2, 5, 16, 23])
def test_window_equals_dense_sdpa_on_the_last_positions(bs, window):
    """Against torch's scaled_dot_product_attention in float64 over the last W
    gathered positions only."""
    lens = [1, window - 1, window, window + 1, 3 * bs + 7, 70]
    w = _small(43 + bs + window, [max(1, L) for L in lens], d=16, bs=bs, poison=True)
    kc, vc = _materialize(w)
    out = _decode_w(w, window, kc=kc, vc=vc)
    st = w.steps[0]
    for s, L in enumerate(st.context_lens.tolist()):
        lo = max(0, L - window)
        ks = torch.stack([_gather(kc, st.block_tables[s], k, L, bs)[lo:] for k in range(2)]).double()
        vs = torch.stack([_gather(vc, st.block_tables[s], k, L, bs)[lo:] for k in range(2)]).double()
        ks = ks.repeat_interleave(2, dim=0)[None]
        vs = vs.repeat_interleave(2, dim=0)[None]
        qs = st.query[s].double()[None, :, None, :]
        ref = torch.nn.functional.scaled_dot_product_attention(qs, ks, vs, scale=w.scale)
        assert torch.allclose(out[s], ref[0, :, 0], rtol=0, atol=1e-12), (s, L)


def test_window_never_reads_blocks_before_it():
    """Blocks wholly before the window may be released: -1 table entries and NaN in
    those blocks give the same output as intact ones, while an entry inside the
    window that is invalid is still reported."""
    w = _small(44, [50, 70, 33], bs=4, poison=True)
    kc, vc = _materialize(w)
    window = 21
    ref = _decode_w(w, window, kc=kc, vc=vc)
    st = w.steps[0]
    bt = st.block_tables.clone()
    kc2, vc2 = kc.clone(), vc.clone()
    for s, L in enumerate(st.context_lens.tolist()):
        first = max(0, L - window) // 4
        for i in range(first):
            b = int(bt[s, i])
            kc2[b] = float("nan")
            vc2[b] = float("nan")
            bt[s, i] = -1
    assert torch.equal(_decode_w(w, window, kc=kc2, vc=vc2, tables=bt), ref)
    s, L = 0, int(st.context_lens[0])
    bt[s, (L - 1) // 4] = -1
    with pytest.raises(ValueError):
        _decode_w(w, window, kc=kc2, vc=vc2, tables=bt)


def test_sliding_window_workload_releases_and_reuses_blocks():
    """The harness releases the blocks that left each window (entries -1), hands them
    out again, keeps the structure consistent, and the oracle never needs them."""
    w = wl.sliding_window_decode(seed=45, num_seqs=6, window=24, block_size=8, num_steps=4,
                                 len_range=(1, 120), poison=True)
    kc, vc = w.key_cache.clone(), w.value_cache.clone()
    for i, st in enumerate(w.steps):
        for L, row in zip(st.context_lens.tolist(), st.block_tables.tolist()):
            first = max(0, L - 24) // 8
            assert all(x == -1 for x in row[:first])
            assert all(x >= 0 for x in row[first:-(-L // 8)])
        out = oracle.run_workload_step(w, i, kc, vc)
        assert torch.isfinite(out).all()
    # the pool is sized for the windows, far below the full contexts
    assert w.num_blocks < sum(-(-int(L) // 8) for L in w.steps[-1].context_lens)


# --- per-head 8-bit scales and the amax report -----------------------------------------

def _fp8_heads(seed=71, spread=3.0):
    return wl.variable_length_decode("h", seed, [1, 9, 40, 77], 8, 4, 16, 8, "e4m3", num_steps=2,
                                     head_spread=spread)


def test_equal_head_scales_are_the_per_tensor_scale():
    """Per-head scales all equal to s give the per-tensor-s bytes and outputs."""
    w = wl.variable_length_decode("t", 72, [3, 17, 50], 8, 4, 16, 8, "e4m3", num_steps=2)
    hk = w.num_kv_heads
    kc1, vc1 = w.key_cache.clone(), w.value_cache.clone()
    kc2, vc2 = w.key_cache.clone(), w.value_cache.clone()
    ksh = torch.full((hk,), w.k_scale)
    vsh = torch.full((hk,), w.v_scale)
    for st in w.steps:
        oracle.reshape_and_cache(st.new_key, st.new_value, kc1, vc1, st.slot_mapping, w.k_scale, w.v_scale)
        oracle.reshape_and_cache(st.new_key, st.new_value, kc2, vc2, st.slot_mapping, 1.0, 1.0, ksh, vsh)
        assert torch.equal(kc1.view(torch.uint8), kc2.view(torch.uint8))
        assert torch.equal(vc1.view(torch.uint8), vc2.view(torch.uint8))
        a = oracle.paged_attention_decode(st.query, kc1, vc1, st.block_tables, st.context_lens, w.scale,
                                          w.k_scale, w.v_scale)
        b = oracle.paged_attention_decode(st.query, kc2, vc2, st.block_tables, st.context_lens, w.scale,
                                          1.0, 1.0, k_head_scales=ksh, v_head_scales=vsh)
        assert torch.equal(a, b)


def test_head_scales_act_head_by_head():
    """With different scales per KV head, the write and the decode equal, bit for bit,
    the per-tensor write and decode run on each KV head alone with its own scale (a
    one-head slice of the cache and of the query group)."""
    w = _fp8_heads()
    hk, g = w.num_kv_heads, w.num_heads // w.num_kv_heads
    assert len(set(w.k_head_scales.tolist())) == hk
    kc, vc = w.key_cache.clone(), w.value_cache.clone()
    for i, st in enumerate(w.steps):
        ref_k, ref_v = kc.clone(), vc.clone()
        out = oracle.run_workload_step(w, i, kc, vc)
        for h in range(hk):
            ks, vs = float(w.k_head_scales[h]), float(w.v_head_scales[h])
            kh, vh = ref_k[:, h:h + 1], ref_v[:, h:h + 1]
            oracle.reshape_and_cache(st.new_key[:, h:h + 1], st.new_value[:, h:h + 1], kh, vh, st.slot_mapping, ks, vs)
            assert torch.equal(kh.view(torch.uint8), kc[:, h:h + 1].view(torch.uint8))
            o = oracle.paged_attention_decode(st.query[:, h * g:(h + 1) * g], kh, vh, st.block_tables,
                                              st.context_lens, w.scale, ks, vs)
            assert torch.equal(o, out[:, h * g:(h + 1) * g])


def test_write_reports_per_head_amax():
    """amax[h] becomes max(amax[h], the largest |x| written for head h), tokens with a
    negative slot excluded; a NaN makes its head's amax NaN and leaves the others."""
    w = _fp8_heads(spread=4.0)
    st = w.steps[0]
    hk = w.num_kv_heads
    kc, vc = w.key_cache.clone(), w.value_cache.clone()
    sm = st.slot_mapping.clone()
    sm[1] = -1
    ka = torch.zeros(hk, dtype=torch.float64)
    va = torch.full((hk,), 0.5, dtype=torch.float64)
    key, value = st.new_key.clone(), st.new_value.clone()
    oracle.reshape_and_cache(key, value, kc, vc, sm, 1.0, 1.0, w.k_head_scales, w.v_head_scales, ka, va)
    keep = sm >= 0
    ek = key[keep].double().abs().amax(dim=(0, 2))
    ev = torch.maximum(value[keep].double().abs().amax(dim=(0, 2)), torch.tensor(0.5, dtype=torch.float64))
    assert torch.equal(ka, ek) and torch.equal(va, ev)
    key[0, 2, 5] = float("nan")
    ka2 = torch.zeros(hk, dtype=torch.float64)
    oracle.reshape_and_cache(key, value, kc, vc, sm, 1.0, 1.0, w.k_head_scales, w.v_head_scales, ka2, None)
    assert torch.isnan(ka2[2]) and torch.equal(ka2[torch.arange(hk) != 2], ek[torch.arange(hk) != 2])


# --- prefill / chunked prefill ------------------------------------------------------------

def _prefill_small(seed=81, prefix=(0, 5, 13, 40), chunk=(7, 1, 20, 9), bs=4, kv="bf16", poison=True):
    return wl.chunked_prefill(seed=seed, prefix_lens=prefix, chunk_lens=chunk, num_heads=4, num_kv_heads=2,
                              head_dim=16, block_size=bs, kv_dtype=kv, poison=poison)


def test_prefill_is_a_chain_of_decodes():
    """Each new token's output equals, bit for bit, decode of one query over the
    context cut at its own position (causal attention is decode at every position)."""
    w = _prefill_small()
    kc, vc = _materialize(w)
    st = w.steps[0]
    out = oracle.paged_attention_prefill(st.query, kc, vc, st.block_tables, st.context_lens, st.query_start_loc,
                                         w.scale)
    qsl = st.query_start_loc.tolist()
    for s, L in enumerate(st.context_lens.tolist()):
        n = qsl[s + 1] - qsl[s]
        for i in range(n):
            row = qsl[s] + i
            ref = oracle.paged_attention_decode(st.query[row:row + 1], kc, vc, st.block_tables[s:s + 1],
                                                torch.tensor([L - n + i + 1], dtype=torch.int32), w.scale)
            assert torch.equal(out[row], ref[0]), (s, i)


@pytest.mark.parametrize("bs", [4, 16])
def test_prefill_equals_causal_sdpa(bs):
    """Against torch's scaled_dot_product_attention in float64 with a causal mask
    shifted by the cached prefix, on the gathered K/V of each sequence."""
    w = _prefill_small(seed=82 + bs, prefix=(0, 3, 16, 33), chunk=(9, 17, 4, 30), bs=bs)
    kc, vc = _materialize(w)
    st = w.steps[0]
    out = oracle.paged_attention_prefill(st.query, kc, vc, st.block_tables, st.context_lens, st.query_start_loc,
                                         w.scale)
    qsl = st.query_start_loc.tolist()
    for s, L in enumerate(st.context_lens.tolist()):
        n = qsl[s + 1] - qsl[s]
        ks = torch.stack([_gather(kc, st.block_tables[s], k, L, bs) for k in range(2)]).double()
        vs = torch.stack([_gather(vc, st.block_tables[s], k, L, bs) for k in range(2)]).double()
        ks = ks.repeat_interleave(2, dim=0)[None]
        vs = vs.repeat_interleave(2, dim=0)[None]
        qs = st.query[qsl[s]:qsl[s + 1]].double().permute(1, 0, 2)[None]     # [1, Hq, n, D]
        mask = torch.arange(L)[None, :] <= (L - n + torch.arange(n))[:, None]
        ref = torch.nn.functional.scaled_dot_product_attention(qs, ks, vs, attn_mask=mask, scale=w.scale)
        assert torch.allclose(out[qsl[s]:qsl[s + 1]], ref[0].permute(1, 0, 2), rtol=0, atol=1e-12), s


def test_prefill_over_an_8bit_cache_equals_causal_sdpa():
    """An e4m3 cache with separate K and V scales: the oracle's prefill equals torch's
    causal scaled_dot_product_attention in float64 over the cache decoded by torch's
    own float8 conversion and scaled (K by its scale, V by its)."""
    w = _prefill_small(seed=87, prefix=(0, 6, 21), chunk=(5, 12, 3), bs=8, kv="e4m3")
    assert w.k_scale != w.v_scale
    kc, vc = _materialize(w)
    st = w.steps[0]
    out = oracle.paged_attention_prefill(st.query, kc, vc, st.block_tables, st.context_lens, st.query_start_loc,
                                         w.scale, w.k_scale, w.v_scale)
    bs = w.block_size

    def gather8(cache, table, L):      # [Hk, L, D] values; torch cannot index fp8 on the CPU
        n = -(-L // bs)
        blocks = cache.view(torch.uint8)[table[:n].long()].view(torch.float8_e4m3fn).double()
        return blocks.permute(1, 0, 2, 3).reshape(blocks.shape[1], n * bs, -1)[:, :L]

    qsl = st.query_start_loc.tolist()
    for s, L in enumerate(st.context_lens.tolist()):
        n = qsl[s + 1] - qsl[s]
        ks = (gather8(kc, st.block_tables[s], L) * w.k_scale).repeat_interleave(2, dim=0)[None]
        vs = (gather8(vc, st.block_tables[s], L) * w.v_scale).repeat_interleave(2, dim=0)[None]
        qs = st.query[qsl[s]:qsl[s + 1]].double().permute(1, 0, 2)[None]
        mask = torch.arange(L)[None, :] <= (L - n + torch.arange(n))[:, None]
        ref = torch.nn.functional.scaled_dot_product_attention(qs, ks, vs, attn_mask=mask, scale=w.scale)
        assert torch.allclose(out[qsl[s]:qsl[s + 1]], ref[0].permute(1, 0, 2), rtol=0, atol=1e-12), s


def test_prefill_of_one_token_is_decode():
    """A chunk of one token per sequence is exactly the decode step."""
    w = _prefill_small(seed=84, prefix=(3, 16, 40), chunk=(1, 1, 1))
    kc, vc = _materialize(w)
    st = w.steps[0]
    pre = oracle.paged_attention_prefill(st.query, kc, vc, st.block_tables, st.context_lens, st.query_start_loc,
                                         w.scale)
    dec = oracle.paged_attention_decode(st.query, kc, vc, st.block_tables, st.context_lens, w.scale)
    assert torch.equal(pre, dec)


def test_prefill_first_token_of_a_prompt_returns_its_value():
    """The first token of a fresh prompt sees only itself: its output is its V."""
    w = _prefill_small(seed=85, prefix=(0, 0), chunk=(5, 12), kv="f32")
    kc, vc = _materialize(w)
    st = w.steps[0]
    out = oracle.paged_attention_prefill(st.query, kc, vc, st.block_tables, st.context_lens, st.query_start_loc,
                                         w.scale)
    for s, q0 in enumerate(st.query_start_loc.tolist()[:-1]):
        for h in range(4):
            v = _gather(vc, st.block_tables[s], h // 2, 1, 4)[0].double()
            assert torch.equal(out[q0, h], v)


def test_prefix_cached_prefill_equals_private_copies():
    """Prompts that share a system prompt's cached blocks (the prefix cache's tables)
    give, bit for bit, the prefill of tables whose blocks were first copied into
    private blocks; the shared blocks are really shared."""
    w = wl.prefix_cached_prefill(seed=12, system_len=70, suffix_lens=(9, 1, 33, 16), num_heads=8,
                                 num_kv_heads=2, head_dim=64, block_size=16, poison=True)
    kc, vc = _materialize(w)
    st = w.steps[0]
    shared = oracle.paged_attention_prefill(st.query, kc, vc, st.block_tables, st.context_lens,
                                            st.query_start_loc, w.scale)
    assert torch.isfinite(shared).all()
    s = st.block_tables.shape[0]
    nblk = [-(-int(L) // w.block_size) for L in st.context_lens]
    kp = torch.full((sum(nblk),) + tuple(kc.shape[1:]), float("nan"), dtype=kc.dtype)
    vp = torch.full_like(kp, float("nan"))
    bt = torch.full((s, st.block_tables.shape[1]), -1, dtype=torch.int32)
    nxt = 0
    for i in range(s):
        for j in range(nblk[i]):
            src = int(st.block_tables[i, j])
            kp[nxt], vp[nxt] = kc[src], vc[src]
            bt[i, j] = nxt
            nxt += 1
    private = oracle.paged_attention_prefill(st.query, kp, vp, bt, st.context_lens, st.query_start_loc, w.scale)
    assert torch.equal(shared, private)
    assert len(set(st.block_tables[:, :4].flatten().tolist())) == 4   # 64 cached tokens: 4 shared blocks
    qsl = st.query_start_loc.tolist()
    assert [qsl[i + 1] - qsl[i] for i in range(s)] == [70 + n - 64 for n in (9, 1, 33, 16)]
