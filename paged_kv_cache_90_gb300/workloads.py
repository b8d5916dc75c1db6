"""Seeded synthetic inputs for the paged decode path.

This module holds no attention arithmetic.  It draws tensors from seeded
``torch.Generator`` streams on the CPU and lays out block tables, slot mappings and
copy-on-write pairs through :mod:`block_manager`.  The GPU kernels and the CPU oracle
are both fed these same tensors.

Shapes follow the workloads the pages describe: a pool of fixed-size blocks with
scattered (shuffled) physical ids, block size 16 by default, Llama-3-8B-like heads
(32 query / 8 KV heads, head_dim 128; gufacode.com "PagedAttention:KV cache 的页表革命",
section "GPU 上 KV cache 池子有多大"), mixed lengths, shared prefixes with parallel
sampling (vasteelab.pages.dev "PagedAttentionとは？", section "負荷試験"), GQA head
sharing and an 8-bit KV cache (ultralytics.com glossary "PagedAttention", section
"관련 기법").

Cache layout: ``[num_blocks, num_kv_heads, block_size, head_dim]``, innermost
contiguous.  The ultralytics.com PyTorch example's pool ``[num_blocks, block_size,
head_dim]`` is its one-head case.
"""
from __future__ import annotations

import math
from dataclasses import dataclass, field
from typing import List, Optional, Sequence

import torch

from .block_manager import BlockAllocator, BlockManager, PrefixCache, blocks_needed, validate_cow_pairs

DTYPES = {"f32": torch.float32, "bf16": torch.bfloat16, "e4m3": torch.float8_e4m3fn}
DTYPE_NAMES = {v: k for k, v in DTYPES.items()}
_E4M3_MAX = 448.0
_CHUNK = 1 << 24


@dataclass
class DecodeStep:
    """Inputs of one decode step: each sequence appends one token, then attends."""
    query: torch.Tensor          # [S, Hq, D]
    new_key: torch.Tensor        # [S, Hk, D] (source dtype: f32 or bf16)
    new_value: torch.Tensor      # [S, Hk, D]
    slot_mapping: torch.Tensor   # [S] int64, slot of each new token
    block_tables: torch.Tensor   # [S, MB] int32, padded with -1
    context_lens: torch.Tensor   # [S] int32, counts the new token
    cow_pairs: torch.Tensor      # [n, 2] int64 (src, dst), copied before the append
    # prefill: query rows of sequence s are query_start_loc[s] .. query_start_loc[s+1]-1
    # (then query, new_key, new_value and slot_mapping hold every new token, packed)
    query_start_loc: Optional[torch.Tensor] = None


@dataclass
class Workload:
    name: str
    num_heads: int
    num_kv_heads: int
    head_dim: int
    block_size: int
    num_blocks: int
    max_blocks_per_seq: int
    scale: float
    k_scale: float
    v_scale: float
    key_cache: torch.Tensor      # initial pool contents [NB, Hk, bs, D]
    value_cache: torch.Tensor
    steps: List[DecodeStep] = field(default_factory=list)
    seed: int = 0
    sliding_window: int = 0      # attend to the last W positions only (0: all)
    k_head_scales: Optional[torch.Tensor] = None   # 8-bit cache: one fp32 scale per KV head
    v_head_scales: Optional[torch.Tensor] = None

    @property
    def num_seqs(self) -> int:
        return int(self.steps[0].query.shape[0])

    @property
    def kv_dtype(self) -> torch.dtype:
        return self.key_cache.dtype

    @property
    def q_dtype(self) -> torch.dtype:
        return self.steps[0].query.dtype


def _randn(shape, dtype: torch.dtype, g: torch.Generator) -> torch.Tensor:
    """N(0, 1) draws rounded to ``dtype``, generated in chunks to bound memory."""
    n = math.prod(shape)
    out = torch.empty(n, dtype=dtype)
    for i in range(0, n, _CHUNK):
        m = min(_CHUNK, n - i)
        out[i:i + m] = torch.randn(m, generator=g, dtype=torch.float32)
    return out.view(*shape)


def _quantize_e4m3(x: torch.Tensor, scale: float) -> torch.Tensor:
    """Pool contents for an 8-bit cache: ``x / scale`` cast by torch's own
    float8_e4m3fn conversion (input generation only)."""
    out = torch.empty(x.shape, dtype=torch.float8_e4m3fn)
    xf, of = x.reshape(-1), out.view(-1)
    for i in range(0, xf.numel(), _CHUNK):
        of[i:i + _CHUNK] = (xf[i:i + _CHUNK].float() / scale).to(torch.float8_e4m3fn)
    return out


def _amax(x: torch.Tensor) -> float:
    xf = x.reshape(-1)
    m = 0.0
    for i in range(0, xf.numel(), _CHUNK):
        m = max(m, float(xf[i:i + _CHUNK].float().abs().max()))
    return m


def _make_pool(nb, hk, bs, d, kv_dtype: str, g: torch.Generator, head_spread: float = 0.0):
    """Random K and V pools (every slot holds N(0,1)-shaped data, used or not).
    ``head_spread`` > 0 (8-bit caches) multiplies KV head h's data by
    2^(head_spread * (h / (hk - 1) - 1/2)) and returns one scale per head (amax / 448)
    as the last two values; otherwise those are None."""
    src = torch.bfloat16 if kv_dtype == "e4m3" else DTYPES[kv_dtype]
    k = _randn((nb, hk, bs, d), src, g)
    v = _randn((nb, hk, bs, d), src, g)
    if kv_dtype != "e4m3":
        return k, v, 1.0, 1.0, None, None
    if head_spread:
        mult = torch.tensor([2.0 ** (head_spread * (h / max(hk - 1, 1) - 0.5)) for h in range(hk)])
        k = (k.float() * mult.view(1, hk, 1, 1)).to(src)
        v = (v.float() * mult.view(1, hk, 1, 1)).to(src)
        ksh = torch.tensor([_amax(k[:, h]) / _E4M3_MAX for h in range(hk)], dtype=torch.float32)
        vsh = torch.tensor([_amax(v[:, h]) / _E4M3_MAX for h in range(hk)], dtype=torch.float32)
        kq = torch.empty(k.shape, dtype=torch.float8_e4m3fn)
        vq = torch.empty(v.shape, dtype=torch.float8_e4m3fn)
        for h in range(hk):
            kq[:, h] = _quantize_e4m3(k[:, h], float(ksh[h]))
            vq[:, h] = _quantize_e4m3(v[:, h], float(vsh[h]))
        return kq, vq, 1.0, 1.0, ksh, vsh
    k_scale = float(torch.tensor(_amax(k) / _E4M3_MAX, dtype=torch.float32))
    v_scale = float(torch.tensor(_amax(v) / _E4M3_MAX, dtype=torch.float32))
    return _quantize_e4m3(k, k_scale), _quantize_e4m3(v, v_scale), k_scale, v_scale, None, None


def _step(mgr: BlockManager, seq_ids: Sequence, g: torch.Generator, hq: int, hk: int,
          d: int, q_dtype: torch.dtype, src_dtype: torch.dtype, mb: int, window: int = 0) -> DecodeStep:
    """Every sequence in ``seq_ids`` appends one token (copy-on-write first if its
    target block is shared; with a sliding window, blocks that left it are released);
    then the step's query and new K/V are drawn."""
    slots, pairs = [], []
    for sid in seq_ids:
        slot, pair = mgr.append_token(sid)
        slots.append(slot)
        if pair is not None:
            pairs.append(pair)
        if window:
            mgr.release_outside_window(sid, window)
    validate_cow_pairs(pairs, mgr.alloc.num_blocks)
    s = len(seq_ids)
    query = _randn((s, hq, d), q_dtype, g)
    new_key = _randn((s, hk, d), src_dtype, g)
    new_value = _randn((s, hk, d), src_dtype, g)
    return DecodeStep(
        query=query, new_key=new_key, new_value=new_value,
        slot_mapping=torch.tensor(slots, dtype=torch.int64),
        block_tables=torch.tensor(mgr.block_table_rows(seq_ids, mb), dtype=torch.int32).view(s, mb),
        context_lens=torch.tensor([mgr.seqs[i].length for i in seq_ids], dtype=torch.int32),
        cow_pairs=torch.tensor(pairs, dtype=torch.int64).view(-1, 2),
    )


def _occupied_slots(mgr: BlockManager) -> torch.Tensor:
    """Flat slot indices that hold a cached token right now."""
    occ = set()
    for s in mgr.seqs.values():
        for pos in range(s.length):
            if s.blocks[pos // mgr.bs] >= 0:  # not released
                occ.add(s.slot(pos, mgr.bs))
    return torch.tensor(sorted(occ), dtype=torch.int64)


def _poison(cache: torch.Tensor, occupied: torch.Tensor) -> None:
    """Overwrite every slot that holds no token with NaN, so that a kernel which
    reads an unused tail slot or an unreferenced block is caught."""
    nb, hk, bs, d = cache.shape
    keep = torch.zeros(nb * bs, dtype=torch.bool)
    keep[occupied] = True
    keep = keep.view(nb, 1, bs, 1).expand(nb, hk, bs, d)
    if cache.dtype == torch.float8_e4m3fn:
        raw = cache.view(torch.uint8)
        raw[~keep] = 0x7F
    else:
        cache[~keep] = float("nan")


def _finish(name, seed, hq, hk, d, bs, nb, mb, kc, vc, ks, vs, steps, scale=None, window=0,
            ksh=None, vsh=None) -> Workload:
    return Workload(name=name, num_heads=hq, num_kv_heads=hk, head_dim=d, block_size=bs,
                    num_blocks=nb, max_blocks_per_seq=mb,
                    scale=float(scale if scale is not None else 1.0 / math.sqrt(d)),
                    k_scale=ks, v_scale=vs, key_cache=kc, value_cache=vc, steps=steps, seed=seed,
                    sliding_window=int(window), k_head_scales=ksh, v_head_scales=vsh)


def variable_length_decode(name: str, seed: int, lengths: Sequence[int], num_heads: int,
                           num_kv_heads: int, head_dim: int, block_size: int, kv_dtype: str,
                           q_dtype: str = "bf16", num_steps: int = 1, pool_slack: float = 0.10,
                           num_blocks: Optional[int] = None, poison: bool = False,
                           scale: Optional[float] = None, window: int = 0,
                           head_spread: float = 0.0) -> Workload:
    """Sequences with the given context lengths *after* the first append.

    The pool holds the needed blocks (for all ``num_steps`` appends) plus
    ``pool_slack`` spare ones, handed out in a seeded random order so every table is a
    scattered set of physical ids.  Each step appends one token per sequence.  With a
    sliding ``window``, blocks wholly before each sequence's window are released (their
    table entries -1; with ``poison`` their slots hold NaN) and may be handed out again.
    ``head_spread`` > 0 with an 8-bit cache gives the KV heads different magnitudes and
    one scale per head.
    """
    g = torch.Generator().manual_seed(seed)
    lengths = [int(x) for x in lengths]
    if min(lengths) < 1:
        raise ValueError("every context length must count the appended token")
    if window:  # a sequence holds its window's blocks, plus one being filled
        need = sum(min(blocks_needed(L + num_steps - 1, block_size), blocks_needed(window, block_size) + 2)
                   for L in lengths)
    else:
        need = sum(blocks_needed(L + num_steps - 1, block_size) for L in lengths)
    nb = num_blocks if num_blocks is not None else int(math.ceil(need * (1.0 + pool_slack)))
    mb = max(blocks_needed(L + num_steps - 1, block_size) for L in lengths)
    perm = torch.randperm(nb, generator=g).tolist()
    mgr = BlockManager(BlockAllocator(nb, block_size, perm))
    seq_ids = list(range(len(lengths)))
    for sid, L in zip(seq_ids, lengths):
        if not window:
            mgr.add_sequence(sid, L - 1)
            continue
        # grow token by token, giving back what leaves the window; positions before the
        # first step's window (L - window, after its append) are released too
        mgr.add_sequence(sid, 0)
        for _ in range(L - 1):
            mgr.append_token(sid)
            mgr.release_outside_window(sid, window - 1)
    kc, vc, ks, vs, ksh, vsh = _make_pool(nb, num_kv_heads, block_size, head_dim, kv_dtype, g, head_spread)
    if poison:
        occ = _occupied_slots(mgr)
        _poison(kc, occ)
        _poison(vc, occ)
    src = torch.bfloat16 if kv_dtype == "e4m3" else DTYPES[kv_dtype]
    steps = [_step(mgr, seq_ids, g, num_heads, num_kv_heads, head_dim, DTYPES[q_dtype], src, mb, window)
             for _ in range(num_steps)]
    if head_spread and ksh is not None:  # the new tokens have their head's magnitude too
        mult = torch.tensor([2.0 ** (head_spread * (h / max(num_kv_heads - 1, 1) - 0.5))
                             for h in range(num_kv_heads)]).view(1, num_kv_heads, 1)
        for st in steps:
            st.new_key = (st.new_key.float() * mult).to(src)
            st.new_value = (st.new_value.float() * mult).to(src)
    mgr.check_structure()
    return _finish(name, seed, num_heads, num_kv_heads, head_dim, block_size, nb, mb,
                   kc, vc, ks, vs, steps, scale, window, ksh, vsh)


# --- the five workloads -----------------------------------------------------------

def tiny(seed: int = 1, poison: bool = True) -> Workload:
    """3 sequences of 5, 17 and 40 tokens, 4 query = 4 KV heads, head_dim 64,
    block size 16, a pool of 64 blocks, fp32 data, scale 1/8."""
    return variable_length_decode("tiny_f32", seed, [5, 17, 40], 4, 4, 64, 16, "f32",
                                  q_dtype="f32", num_blocks=64, poison=poison)


def scalar_example(physical: Sequence[int] = (4, 1), num_blocks: int = 8,
                   head_dim: int = 1, dtype: str = "f32") -> Workload:
    """The pages' scalar case: one head, keys 0, query 1, values 1..5, four tokens
    per block, logical blocks 0 and 1 at the given physical blocks
    (paweldubiel.com "PagedAttention", sections "Mecanismo y detalles" and
    "El orden del texto no es la dirección de memoria").  ``head_dim`` > 1 pads the
    head with zeros: q.k is unchanged and every extra output column is 0."""
    bs, L = 4, 5
    dt = DTYPES[dtype]
    kc = torch.zeros(num_blocks, 1, bs, head_dim, dtype=dt)
    vc = torch.zeros(num_blocks, 1, bs, head_dim, dtype=dt)
    for pos in range(L):
        vc[physical[pos // bs], 0, pos % bs, 0] = float(pos + 1)
    q = torch.zeros(1, 1, head_dim, dtype=dt)
    q[0, 0, 0] = 1.0
    mb = len(physical)
    step = DecodeStep(
        query=q, new_key=torch.zeros(0, 1, head_dim, dtype=dt),
        new_value=torch.zeros(0, 1, head_dim, dtype=dt),
        slot_mapping=torch.zeros(0, dtype=torch.int64),
        block_tables=torch.tensor([list(physical)], dtype=torch.int32),
        context_lens=torch.tensor([L], dtype=torch.int32),
        cow_pairs=torch.zeros(0, 2, dtype=torch.int64))
    return Workload(name="scalar_example", num_heads=1, num_kv_heads=1, head_dim=head_dim,
                    block_size=bs, num_blocks=num_blocks, max_blocks_per_seq=mb, scale=1.0,
                    k_scale=1.0, v_scale=1.0, key_cache=kc, value_cache=vc, steps=[step])


def llama3_8b_decode(seed: int = 2, num_seqs: int = 64, len_range=(128, 2048),
                     block_size: int = 16, kv_dtype: str = "bf16", poison: bool = False) -> Workload:
    """Llama-3-8B-shaped decode layer: ``num_seqs`` sequences whose cached lengths are
    uniform in ``len_range``; one new token each; 32/8 heads, head_dim 128."""
    g = torch.Generator().manual_seed(seed)
    old = torch.randint(len_range[0], len_range[1] + 1, (num_seqs,), generator=g).tolist()
    return variable_length_decode(f"llama3_8b_decode_s{num_seqs}_bs{block_size}_{kv_dtype}",
                                  seed, [L + 1 for L in old], 32, 8, 128, block_size, kv_dtype,
                                  poison=poison)


def long_context(seed: int = 3, block_size: int = 16, num_seqs: int = 8,
                 context_len: int = 32768, poison: bool = False) -> Workload:
    """Long-context decode: every sequence holds ``context_len`` tokens after its
    append; 32/8 heads, head_dim 128, bf16."""
    return variable_length_decode(f"long_context_s{num_seqs}_L{context_len}_bs{block_size}",
                                  seed, [context_len] * num_seqs, 32, 8, 128, block_size, "bf16",
                                  poison=poison)


def continuous_batching(seed: int = 5, block_size: int = 16, kv_dtype: str = "bf16",
                        num_seqs: int = 256, num_steps: int = 10, median: float = 512.0,
                        sigma: float = 1.0, cap: int = 8192, poison: bool = False,
                        head_spread: float = 0.0) -> Workload:
    """Continuous-batching mix: lengths round(lognormal(ln median, sigma)) clamped to
    [1, cap], ``num_steps`` decode steps each appending one token per sequence (a new
    block is taken whenever a sequence's last block is full).  ``head_spread`` > 0 with
    an 8-bit cache: KV heads of different magnitudes, one scale per head."""
    g = torch.Generator().manual_seed(seed)
    z = torch.randn(num_seqs, generator=g, dtype=torch.float64)
    lens = torch.exp(math.log(median) + sigma * z).round().clamp(1, cap).long().tolist()
    return variable_length_decode(f"continuous_batching_s{num_seqs}_bs{block_size}_{kv_dtype}",
                                  seed, lens, 32, 8, 128, block_size, kv_dtype,
                                  num_steps=num_steps, poison=poison, head_spread=head_spread)


def shared_prefix_cow(seed: int = 4, num_groups: int = 32, group_size: int = 4,
                      prefix_blocks: int = 64, suffix_range=(16, 512), block_size: int = 16,
                      pool_slack: float = 0.10, poison: bool = False) -> Workload:
    """Shared prefix + parallel sampling with copy-on-write.

    Every sequence's table starts with the same ``prefix_blocks`` physical blocks.
    Each group of ``group_size`` samples shares a suffix of ``u`` tokens, u uniform in
    ``suffix_range`` and not a multiple of the block size, so the group's last block is
    partly filled and shared.  The step appends one token to every sample: the first
    ``group_size - 1`` writers of a group get a private copy of that block (the copy
    pairs of the step), the last one writes in place.
    """
    g = torch.Generator().manual_seed(seed)
    us = []
    while len(us) < num_groups:
        u = int(torch.randint(suffix_range[0], suffix_range[1] + 1, (1,), generator=g))
        if u % block_size:
            us.append(u)
    need = prefix_blocks + sum(blocks_needed(u, block_size) + group_size - 1 for u in us)
    nb = int(math.ceil(need * (1.0 + pool_slack)))
    perm = torch.randperm(nb, generator=g).tolist()
    mgr = BlockManager(BlockAllocator(nb, block_size, perm))
    mgr.add_sequence("prefix", prefix_blocks * block_size)
    seq_ids = []
    for gi, u in enumerate(us):
        head = (gi, 0)
        mgr.fork("prefix", head)
        for _ in range(u):
            _, pair = mgr.append_token(head)
            assert pair is None
        seq_ids.append(head)
        for j in range(1, group_size):
            mgr.fork(head, (gi, j))
            seq_ids.append((gi, j))
    mgr.free_sequence("prefix")
    mb = prefix_blocks + max(blocks_needed(u + 1, block_size) for u in us)
    kc, vc, ks, vs, _, _ = _make_pool(nb, 8, block_size, 128, "bf16", g)
    if poison:
        occ = _occupied_slots(mgr)
        _poison(kc, occ)
        _poison(vc, occ)
    step = _step(mgr, seq_ids, g, 32, 8, 128, torch.bfloat16, torch.bfloat16, mb)
    mgr.check_structure()
    return _finish(f"shared_prefix_cow_g{num_groups}x{group_size}", seed, 32, 8, 128, block_size,
                   nb, mb, kc, vc, ks, vs, [step])


def sliding_window_decode(seed: int = 6, num_seqs: int = 8, context_len: int = 32768, window: int = 4096,
                          block_size: int = 16, kv_dtype: str = "bf16", num_steps: int = 1,
                          len_range=None, poison: bool = False) -> Workload:
    """Decode of a sliding-window layer: sequences of ``context_len`` tokens (or lengths
    uniform in ``len_range``) attend to their last ``window`` positions; the blocks
    before each window are released.  32/8 heads, head_dim 128."""
    g = torch.Generator().manual_seed(seed)
    if len_range is not None:
        lens = (torch.randint(len_range[0], len_range[1] + 1, (num_seqs,), generator=g) + 1).tolist()
    else:
        lens = [context_len] * num_seqs
    return variable_length_decode(f"sliding_window_s{num_seqs}_W{window}_bs{block_size}_{kv_dtype}", seed,
                                  lens, 32, 8, 128, block_size, kv_dtype, num_steps=num_steps,
                                  poison=poison, window=window)


def chunked_prefill(seed: int = 7, prefix_lens: Sequence[int] = (0, 0, 512, 1536),
                    chunk_lens: Sequence[int] = (2048, 1024, 512, 512), num_heads: int = 32,
                    num_kv_heads: int = 8, head_dim: int = 128, block_size: int = 16,
                    kv_dtype: str = "bf16", pool_slack: float = 0.10, poison: bool = False) -> Workload:
    """Prefill of prompts (prefix 0) and of later chunks of long prompts: sequence s has
    ``prefix_lens[s]`` tokens cached and appends ``chunk_lens[s]`` new ones, whose K/V
    the step writes and whose queries attend causally to everything before them.  The
    step's query, new K/V and slot mapping hold all new tokens packed, sequence by
    sequence (``query_start_loc``)."""
    g = torch.Generator().manual_seed(seed)
    prefix = [int(x) for x in prefix_lens]
    chunk = [int(x) for x in chunk_lens]
    if len(prefix) != len(chunk) or min(chunk) < 1 or min(prefix) < 0:
        raise ValueError("one prefix and one chunk of >= 1 token per sequence")
    need = sum(blocks_needed(a + b, block_size) for a, b in zip(prefix, chunk))
    nb = int(math.ceil(need * (1.0 + pool_slack))) + 1
    mb = max(blocks_needed(a + b, block_size) for a, b in zip(prefix, chunk))
    perm = torch.randperm(nb, generator=g).tolist()
    mgr = BlockManager(BlockAllocator(nb, block_size, perm))
    seq_ids = list(range(len(prefix)))
    for sid, a in zip(seq_ids, prefix):
        mgr.add_sequence(sid, a)
    kc, vc, ks, vs, _, _ = _make_pool(nb, num_kv_heads, block_size, head_dim, kv_dtype, g)
    if poison:
        # the chunk's slots are written by the step; everything else unused is NaN
        occ = _occupied_slots(mgr)
        _poison(kc, occ)
        _poison(vc, occ)
    slots = []
    for sid, c in zip(seq_ids, chunk):
        for _ in range(c):
            slot, pair = mgr.append_token(sid)
            assert pair is None
            slots.append(slot)
    t = sum(chunk)
    src = torch.bfloat16 if kv_dtype == "e4m3" else DTYPES[kv_dtype]
    q_dtype = torch.float32 if kv_dtype == "f32" else torch.bfloat16
    qsl = [0]
    for c in chunk:
        qsl.append(qsl[-1] + c)
    step = DecodeStep(
        query=_randn((t, num_heads, head_dim), q_dtype, g),
        new_key=_randn((t, num_kv_heads, head_dim), src, g),
        new_value=_randn((t, num_kv_heads, head_dim), src, g),
        slot_mapping=torch.tensor(slots, dtype=torch.int64),
        block_tables=torch.tensor(mgr.block_table_rows(seq_ids, mb), dtype=torch.int32).view(len(seq_ids), mb),
        context_lens=torch.tensor([a + b for a, b in zip(prefix, chunk)], dtype=torch.int32),
        cow_pairs=torch.zeros(0, 2, dtype=torch.int64),
        query_start_loc=torch.tensor(qsl, dtype=torch.int32))
    mgr.check_structure()
    return _finish(f"chunked_prefill_s{len(chunk)}_T{t}_bs{block_size}_{kv_dtype}", seed, num_heads,
                   num_kv_heads, head_dim, block_size, nb, mb, kc, vc, ks, vs, [step])


def prefix_cached_prefill(seed: int = 10, system_len: int = 700, suffix_lens: Sequence[int] = (90, 1, 300, 17, 64),
                          num_heads: int = 32, num_kv_heads: int = 8, head_dim: int = 128, block_size: int = 16,
                          kv_dtype: str = "bf16", poison: bool = False) -> Workload:
    """Prompts that share a system prompt, through the prefix cache: an earlier request
    computed the system prompt (its K/V are in the pool, its full blocks identified, the
    request gone), then each prompt (system prompt + its own suffix) shares the cached
    full blocks and prefills only the rest — one chunked-prefill step whose sequences
    all read the same physical prefix blocks."""
    g = torch.Generator().manual_seed(seed)
    suffix = [int(x) for x in suffix_lens]
    if min(suffix) < 1 or system_len < 1:
        raise ValueError("a system prompt and at least one suffix token per prompt")
    vocab = 32000
    system = torch.randint(0, vocab, (system_len,), generator=g).tolist()
    prompts = [system + torch.randint(0, vocab, (n,), generator=g).tolist() for n in suffix]
    need = blocks_needed(system_len + 1, block_size) + sum(blocks_needed(len(t), block_size) for t in prompts)
    nb = need + 8
    perm = torch.randperm(nb, generator=g).tolist()
    mgr = BlockManager(BlockAllocator(nb, block_size, perm))
    cache = PrefixCache(mgr)
    cache.add_prompt("earlier", system + [0])   # computed before this step; its K/V are the pool's
    kc, vc, ks, vs, _, _ = _make_pool(nb, num_kv_heads, block_size, head_dim, kv_dtype, g)
    mgr.free_sequence("earlier")                # the cache keeps its full blocks
    seq_ids = list(range(len(prompts)))
    slots, chunk = [], []
    for sid, t in zip(seq_ids, prompts):
        sl, cached = cache.add_prompt(sid, t)
        slots += sl
        chunk.append(len(t) - cached)
    mgr.check_structure(held=cache.held())
    if poison:
        # the step writes the new tokens' slots; the shared prefix blocks hold the
        # earlier request's K/V; everything else unused is NaN
        occ = _occupied_slots(mgr)
        new = torch.tensor(slots, dtype=torch.int64)
        keep = occ[~torch.isin(occ, new)]
        _poison(kc, keep)
        _poison(vc, keep)
    mb = max(blocks_needed(len(t), block_size) for t in prompts)
    tq = sum(chunk)
    src = torch.bfloat16 if kv_dtype == "e4m3" else DTYPES[kv_dtype]
    q_dtype = torch.float32 if kv_dtype == "f32" else torch.bfloat16
    qsl = [0]
    for c in chunk:
        qsl.append(qsl[-1] + c)
    step = DecodeStep(
        query=_randn((tq, num_heads, head_dim), q_dtype, g),
        new_key=_randn((tq, num_kv_heads, head_dim), src, g),
        new_value=_randn((tq, num_kv_heads, head_dim), src, g),
        slot_mapping=torch.tensor(slots, dtype=torch.int64),
        block_tables=torch.tensor(mgr.block_table_rows(seq_ids, mb), dtype=torch.int32).view(len(seq_ids), mb),
        context_lens=torch.tensor([len(t) for t in prompts], dtype=torch.int32),
        cow_pairs=torch.zeros(0, 2, dtype=torch.int64),
        query_start_loc=torch.tensor(qsl, dtype=torch.int32))
    return _finish(f"prefix_cached_prefill_s{len(prompts)}_sys{system_len}_bs{block_size}_{kv_dtype}", seed,
                   num_heads, num_kv_heads, head_dim, block_size, nb, mb, kc, vc, ks, vs, [step])


WORKLOADS = {
    "tiny": tiny,
    "llama3_8b_decode": llama3_8b_decode,
    "long_context": long_context,
    "shared_prefix_cow": shared_prefix_cow,
    "continuous_batching": continuous_batching,
    "sliding_window": sliding_window_decode,
    "chunked_prefill": chunked_prefill,
    "prefix_cached_prefill": prefix_cached_prefill,
}
