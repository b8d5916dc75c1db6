"""The seeded inputs both sides run on (CPU): every generated step is a well-formed
paged step — the properties the kernels and the oracle assume rather than check."""
import pytest
import torch

from paged_kv_cache_90_gb300 import workloads as wl


def _small_workloads():
    return [
        wl.tiny(),
        wl.llama3_8b_decode(seed=21, num_seqs=6, len_range=(1, 300)),
        wl.llama3_8b_decode(),                                  # the full-size benchmark batch
        wl.long_context(seed=22, block_size=32, num_seqs=2, context_len=700),
        wl.continuous_batching(seed=23, block_size=8, kv_dtype="e4m3", num_seqs=10, num_steps=4, median=40),
        wl.continuous_batching(seed=24, block_size=16, kv_dtype="bf16", num_seqs=10, num_steps=3, median=40,
                               head_spread=3.0),
        wl.shared_prefix_cow(seed=25, num_groups=3, group_size=4, prefix_blocks=2),
        wl.sliding_window_decode(seed=26, num_seqs=3, context_len=300, window=40),
        wl.chunked_prefill(seed=27, prefix_lens=[0, 30, 100], chunk_lens=[17, 1, 64]),
        wl.prefix_cached_prefill(seed=28, system_len=70, suffix_lens=[5, 1, 33]),
    ]


@pytest.mark.parametrize("w", _small_workloads(), ids=lambda w: w.name)
def test_steps_are_well_formed(w):
    nb, hk, bs, d = w.key_cache.shape
    assert w.value_cache.shape == w.key_cache.shape and hk == w.num_kv_heads and bs == w.block_size
    assert w.num_heads % hk == 0 and d == w.head_dim and nb == w.num_blocks
    for st in w.steps:
        S = st.block_tables.shape[0]
        assert st.block_tables.dtype == torch.int32 and st.context_lens.dtype == torch.int32
        assert st.slot_mapping.dtype == torch.int64 and st.cow_pairs.dtype == torch.int64
        assert st.block_tables.shape[1] == w.max_blocks_per_seq and st.context_lens.shape == (S,)
        L = st.context_lens.long()
        assert (L >= 0).all() and (L <= w.max_blocks_per_seq * bs).all()
        # every attended position's block is a real block of the pool
        W = w.sliding_window
        for s in range(S):
            n = int(L[s])
            first = n - W if (W > 0 and n > W) else 0
            for blk in range(first // bs, -(-n // bs)):
                e = int(st.block_tables[s, blk])
                assert 0 <= e < nb, (s, blk, e)
        # new tokens: distinct slots, each the slot of its position through the table
        slots = st.slot_mapping[st.slot_mapping >= 0]
        assert slots.unique().numel() == slots.numel()
        assert (slots < nb * bs).all()
        if st.query_start_loc is None:
            assert st.query.shape == (S, w.num_heads, d)
            pos = L - 1
            for s in range(S):
                if int(st.slot_mapping[s]) >= 0 and int(L[s]) > 0:
                    want = int(st.block_tables[s, int(pos[s]) // bs]) * bs + int(pos[s]) % bs
                    assert int(st.slot_mapping[s]) == want, s
        else:
            qsl = st.query_start_loc.long()
            assert qsl.shape == (S + 1,) and int(qsl[0]) == 0 and int(qsl[-1]) == st.query.shape[0]
            for s in range(S):
                n_new = int(qsl[s + 1] - qsl[s])
                assert 0 <= n_new <= int(L[s])
                for i in range(n_new):
                    p = int(L[s]) - n_new + i
                    t = int(qsl[s]) + i
                    want = int(st.block_tables[s, p // bs]) * bs + p % bs
                    assert int(st.slot_mapping[t]) == want, (s, i)
        # copy-on-write pairs: distinct destinations, none of them a source
        if st.cow_pairs.numel():
            src, dst = st.cow_pairs[:, 0], st.cow_pairs[:, 1]
            assert dst.unique().numel() == dst.numel()
            assert not (set(dst.tolist()) & set(src.tolist()))
            assert ((src >= 0) & (src < nb) & (dst >= 0) & (dst < nb)).all()


def test_generators_are_seeded():
    a, b = wl.llama3_8b_decode(seed=31, num_seqs=4), wl.llama3_8b_decode(seed=31, num_seqs=4)
    c = wl.llama3_8b_decode(seed=32, num_seqs=4)
    assert torch.equal(a.steps[0].query, b.steps[0].query) and torch.equal(a.key_cache, b.key_cache)
    assert torch.equal(a.steps[0].block_tables, b.steps[0].block_tables)
    assert not torch.equal(a.steps[0].query, c.steps[0].query)
