"""The C ABI without a GPU: the library builds and loads, exports every function
include/pkv.h declares, and its host-side argument checks accept good descriptors
and reject bad ones (dry-run mode: validation only, nothing touches the GPU)."""
import ctypes
import re
from pathlib import Path

import pytest
import torch

from paged_kv_cache_90_gb300 import binding
from paged_kv_cache_90_gb300 import build as pkv_build

HEADER = Path(__file__).resolve().parent.parent / "include" / "pkv.h"


@pytest.fixture(scope="module")
def lib():
    pkv_build.build()
    return binding.load_library()


@pytest.fixture
def dry(lib):
    binding.set_option("dry_run", 1)
    yield lib
    binding.set_option("dry_run", 0)
    binding.set_option("partition_tokens", 0)


def declared_functions():
    text = HEADER.read_text()
    text = re.sub(r"/\*.*?\*/", "", text, flags=re.S)
    return sorted(set(re.findall(r"\b(pkv_[a-z_0-9]+)\s*\(", text)))


def test_exports_every_declared_function(lib):
    names = declared_functions()
    assert {"pkv_paged_attention_decode", "pkv_reshape_and_cache", "pkv_copy_blocks"} <= set(names)
    for n in names:
        assert hasattr(lib, n), f"{n} is declared in pkv.h but not exported"
    assert binding.abi_version() == 3


def _decode_args(S=3, Hq=8, Hk=2, D=128, bs=16, NB=20, MB=4, dtype=torch.bfloat16, kv=torch.bfloat16):
    q = torch.zeros(S, Hq, D, dtype=dtype)
    return dict(out=torch.empty_like(q), query=q,
                key_cache=torch.zeros(NB, Hk, bs, D, dtype=kv), value_cache=torch.zeros(NB, Hk, bs, D, dtype=kv),
                block_tables=torch.zeros(S, MB, dtype=torch.int32), context_lens=torch.ones(S, dtype=torch.int32),
                num_kv_heads=Hk, scale=D ** -0.5, block_size=bs, max_blocks_per_seq=MB)


def _status(fn, **kw):
    try:
        fn(**kw)
        return 0
    except binding.PkvError as e:
        assert e.message, "a failing call must leave a message"
        return e.status


def test_decode_step_validation(dry):
    """The joint write + decode call checks the arguments of both before queueing."""
    def args(**over):
        a = _decode_args()
        T, Hk, D = 3, 2, 128
        a.update(key=torch.zeros(T, Hk, D, dtype=torch.bfloat16), value=torch.zeros(T, Hk, D, dtype=torch.bfloat16),
                 slot_mapping=torch.arange(T, dtype=torch.int64))
        a.update(over)
        return a
    assert _status(binding.decode_step, **args()) == 0
    assert _status(binding.decode_step, **args(slot_mapping=torch.arange(3, dtype=torch.int32))) == 2  # write side
    assert _status(binding.decode_step, **args(key=torch.zeros(3, 2, 64, dtype=torch.bfloat16),
                                               value=torch.zeros(3, 2, 64, dtype=torch.bfloat16))) == 1
    assert _status(binding.decode_step, **args(num_kv_heads=3)) == 1                               # decode side
    assert _status(binding.decode_step, **args(block_size=8)) == 1
    empty = torch.zeros(0, 2, 128, dtype=torch.bfloat16)
    assert _status(binding.decode_step, **args(key=empty, value=empty,
                                               slot_mapping=torch.zeros(0, dtype=torch.int64))) == 0
    assert _status(binding.decode_append, **args()) == 0                        # one token per sequence
    two = torch.zeros(2, 2, 128, dtype=torch.bfloat16)
    assert _status(binding.decode_append, **args(key=two, value=two,
                                                 slot_mapping=torch.arange(2, dtype=torch.int64))) == 1


def test_prepared_step_checks_like_the_call(dry):
    """A prepared step call (arguments marshalled once) checks them at every call and
    gives the status pkv_decode_step gives for the same arguments; it returns `out` and
    keeps its tensors referenced."""
    def args(**over):
        a = _decode_args()
        a.update(key=torch.zeros(3, 2, 128, dtype=torch.bfloat16), value=torch.zeros(3, 2, 128, dtype=torch.bfloat16),
                 slot_mapping=torch.arange(3, dtype=torch.int64))
        a.update(over)
        return a
    for over in ({}, {"slot_mapping": torch.arange(3, dtype=torch.int32)}, {"num_kv_heads": 3},
                 {"block_size": 8}, {"query": torch.zeros(3, 8, 64, dtype=torch.bfloat16)}):
        a = args(**over)
        want = _status(binding.decode_step, **a)
        step = binding.prepare_decode_step(**a)
        for _ in range(2):
            assert _status(step) == want, over
        if want == 0:
            assert step() is a["out"]
    a = args()
    step = binding.prepare_decode_step(**a)
    assert step.tensors[0] is a["out"] and step.tensors[5] is a["key_cache"] and step.tensors[8] is a["context_lens"]


def test_head_scales_and_amax_validation(dry):
    """Per-head scales belong to 8-bit caches only and must be 4-byte aligned; the
    per-tensor scale is not checked when they are given; amax arrays must be aligned."""
    hs = torch.ones(2, dtype=torch.float32)
    a = _decode_args(kv=torch.float8_e4m3fn)
    assert _status(binding.paged_attention_decode, **a, k_head_scales=hs, v_head_scales=hs) == 0
    assert _status(binding.paged_attention_decode, **a, k_scale=0.0, v_scale=0.0, k_head_scales=hs,
                   v_head_scales=hs) == 0
    assert _status(binding.paged_attention_decode, **_decode_args(), k_head_scales=hs) == 1   # bf16 cache
    lib = binding.load_library()
    descs = [binding.describe(a[k]) for k in ("out", "query")]
    kc = binding.describe(a["key_cache"], 1.0)
    kc.head_scales = hs.data_ptr() + 2
    descs += [kc, binding.describe(a["value_cache"], 1.0), binding.describe(a["block_tables"]),
              binding.describe(a["context_lens"])]
    rc = lib.pkv_paged_attention_decode(*[ctypes.byref(x) for x in descs], 2, 0.1, 16, 4, None)
    assert rc == 1 and b"aligned" in lib.pkv_last_error()
    T = 3
    w = [binding.describe(torch.zeros(T, 2, 128, dtype=torch.bfloat16)) for _ in range(2)]
    c = [binding.describe(torch.zeros(20, 2, 16, 128, dtype=torch.float8_e4m3fn), 0.5) for _ in range(2)]
    sm = binding.describe(torch.arange(T, dtype=torch.int64))
    amax = torch.zeros(4, dtype=torch.float32)
    args = [ctypes.byref(x) for x in (w[0], w[1], c[0], c[1], sm)]
    assert lib.pkv_reshape_and_cache_amax(*args, ctypes.c_void_p(amax.data_ptr()), None, None) == 0
    assert lib.pkv_reshape_and_cache_amax(*args, ctypes.c_void_p(amax.data_ptr() + 2), None, None) == 1


def test_decode_validation(dry):
    ok = _decode_args()
    assert _status(binding.paged_attention_decode, **ok) == 0
    assert _status(binding.paged_attention_decode, **ok, sliding_window=5) == 0
    assert _status(binding.paged_attention_decode, **ok, sliding_window=-3) == 1
    assert _status(binding.paged_attention_decode, **_decode_args(kv=torch.float8_e4m3fn),
                   k_scale=0.01, v_scale=0.02) == 0
    assert _status(binding.paged_attention_decode, **_decode_args(dtype=torch.float32, kv=torch.float32, D=64)) == 0
    bad = []
    a = _decode_args(); a["num_kv_heads"] = 3; bad.append((a, 1))                 # != cache heads
    a = _decode_args(Hq=6, Hk=4); bad.append((a, 1))                              # Hq % Hk
    a = _decode_args(); a["block_size"] = 8; bad.append((a, 1))                   # != cache bs
    a = _decode_args(); a["max_blocks_per_seq"] = 5; bad.append((a, 1))           # != table width
    a = _decode_args(D=96); bad.append((a, 2))                                    # head_dim
    a = _decode_args(bs=64); bad.append((a, 2))                                   # block size
    a = _decode_args(); a["out"] = torch.empty(3, 8, 128, dtype=torch.float32); bad.append((a, 1))
    a = _decode_args(); a["block_tables"] = a["block_tables"].long(); bad.append((a, 2))
    a = _decode_args(); a["context_lens"] = torch.ones(2, dtype=torch.int32); bad.append((a, 1))
    a = _decode_args(); a["value_cache"] = torch.zeros(20, 2, 16, 128, dtype=torch.float32); bad.append((a, 1))
    a = _decode_args(); a["query"] = a["query"].transpose(1, 2).contiguous().transpose(1, 2); bad.append((a, 1))
    a = _decode_args(kv=torch.float8_e4m3fn); bad.append((dict(a, k_scale=0.0), 1))  # fp8 scale
    a = _decode_args(); a["scale"] = float("inf"); bad.append((a, 1))
    for args, want in bad:
        extra = {}
        if "k_scale" in args:
            extra["k_scale"] = args.pop("k_scale")
        assert _status(binding.paged_attention_decode, **args, **extra) == want, args


def test_decode_rejects_misaligned_cache(dry):
    a = _decode_args()
    big = torch.zeros(20 * 2 * 16 * 128 + 4, dtype=torch.bfloat16)
    a["key_cache"] = big[1:1 + 20 * 2 * 16 * 128].view(20, 2, 16, 128)   # 2-byte offset
    a["value_cache"] = big[1:1 + 20 * 2 * 16 * 128].view(20, 2, 16, 128)
    assert _status(binding.paged_attention_decode, **a) == 1


def test_cache_views_with_block_stride(dry):
    """K and V as views of one [NB, 2, Hk, bs, D] tensor: strided blocks are fine."""
    a = _decode_args()
    both = torch.zeros(20, 2, 2, 16, 128, dtype=torch.bfloat16)
    a["key_cache"], a["value_cache"] = both[:, 0], both[:, 1]
    assert _status(binding.paged_attention_decode, **a) == 0


def test_reshape_and_cache_validation(dry):
    kc = torch.zeros(10, 2, 16, 128, dtype=torch.bfloat16)
    k = torch.zeros(4, 2, 128, dtype=torch.bfloat16)
    sm = torch.zeros(4, dtype=torch.int64)
    assert _status(binding.reshape_and_cache, key=k, value=k, key_cache=kc, value_cache=kc, slot_mapping=sm) == 0
    f8 = torch.zeros(10, 2, 16, 128, dtype=torch.float8_e4m3fn)
    assert _status(binding.reshape_and_cache, key=k, value=k, key_cache=f8, value_cache=f8,
                   slot_mapping=sm, k_scale=0.5, v_scale=0.5) == 0
    assert _status(binding.reshape_and_cache, key=k.float(), value=k.float(), key_cache=kc, value_cache=kc,
                   slot_mapping=sm) == 2                                            # f32 -> bf16
    assert _status(binding.reshape_and_cache, key=k, value=k, key_cache=kc, value_cache=kc,
                   slot_mapping=sm.int()) == 2                                      # slot dtype
    assert _status(binding.reshape_and_cache, key=k, value=k, key_cache=kc, value_cache=kc,
                   slot_mapping=sm[:3]) == 1                                        # count
    assert _status(binding.reshape_and_cache, key=k[:, :1], value=k[:, :1], key_cache=kc, value_cache=kc,
                   slot_mapping=sm) == 1                                            # heads


def test_copy_blocks_validation(dry):
    c = torch.zeros(10, 2, 16, 128, dtype=torch.bfloat16)
    assert _status(binding.copy_blocks, cache=c, src_dst_pairs=torch.zeros(3, 2, dtype=torch.int64)) == 0
    assert _status(binding.copy_blocks, cache=c, src_dst_pairs=torch.zeros(0, 2, dtype=torch.int64)) == 0
    assert _status(binding.copy_blocks, cache=c, src_dst_pairs=torch.zeros(3, 3, dtype=torch.int64)) == 1
    assert _status(binding.copy_blocks, cache=c, src_dst_pairs=torch.zeros(3, 2, dtype=torch.int32)) == 2


def test_options_and_workspace_size(lib):
    with pytest.raises(binding.PkvError):
        binding.set_option("partition_tokens", 100)
    binding.set_option("partition_tokens", 1024)
    assert binding.get_option("partition_tokens") == 1024
    binding.set_option("partition_tokens", 0)
    # an upper bound over both decode kernels: at least the CUDA-core kernel's partials
    # (8 sequences x 32 heads x 64 partitions of 512 tokens) and the tensor-core kernel's
    # (one slot of 4 heads per warp, per run-time unit and per row)
    big = binding.decode_workspace_bytes(8, 32, 8, 128, 16, 2048)
    assert big >= 8 * 32 * 64 * 130 * 4
    assert big >= (8 * 32) * 130 * 4
    # a short context: no CUDA-core partials, only the tensor-core kernel's slots
    small = binding.decode_workspace_bytes(8, 32, 8, 128, 16, 16)
    assert small >= (8 * 32) * 130 * 4 and small <= big
    assert binding.decode_workspace_bytes(0, 32, 8, 128, 16, 2048) == 0
    assert binding.decode_workspace_bytes(8, 32, 5, 128, 16, 2048) == 0
    # 3 heads per KV head: rows of one head on the tensor path (slots of 1 head)
    assert binding.decode_workspace_bytes(8, 6, 2, 128, 16, 16) >= (8 * 6) * 130 * 4
    for name, bad in (("dynamic_share", 1025), ("dynamic_share", -2), ("dynamic_chunk", 0), ("dynamic_chunk", 65),
                      ("fused_append", -1), ("fused_append", 3)):
        with pytest.raises(binding.PkvError):
            binding.set_option(name, bad)
    assert binding.get_option("dynamic_share") == -1     # automatic
    binding.set_option("dynamic_share", 512)
    assert binding.get_option("dynamic_share") == 512
    binding.set_option("dynamic_share", -1)
    assert binding.get_option("dynamic_chunk") == 4
    assert binding.get_option("fused_append") == 0       # automatic
    with pytest.raises(KeyError):
        binding.set_option("nope", 1)
    assert lib.pkv_set_option(99, 0) == 1


def _raw_decode(lib, descs, num_kv_heads=2, scale=0.1, block_size=16, mb=4):
    ptrs = [None if d is None else ctypes.byref(d) for d in descs]
    return lib.pkv_paged_attention_decode(*ptrs, num_kv_heads, scale, block_size, mb, None)


def test_descriptor_checks(dry):
    """Malformed descriptors fail with INVALID_ARG (or UNSUPPORTED for a known but
    unsupported dtype) and a message naming the argument, before anything is queued."""
    lib = binding.load_library()
    a = _decode_args()
    names = ("out", "query", "key_cache", "value_cache", "block_tables", "context_lens")

    def descs():
        return [binding.describe(a[n]) for n in names]

    assert _raw_decode(lib, descs()) == 0
    for i, n in enumerate(names):
        d = descs()
        d[i] = None                                           # null descriptor
        assert _raw_decode(lib, d) == 1 and n.encode() in lib.pkv_last_error()
        d = descs()
        d[i].data = None                                      # null data pointer
        assert _raw_decode(lib, d) == 1 and n.encode() in lib.pkv_last_error()
        d = descs()
        d[i].dtype = 17                                       # unknown dtype code
        assert _raw_decode(lib, d) == 1 and b"unknown dtype" in lib.pkv_last_error()
        d = descs()
        d[i].ndim = d[i].ndim + 1 if d[i].ndim < 4 else 3     # wrong rank
        assert _raw_decode(lib, d) == 1
        d = descs()
        d[i].shape[0] = -1                                    # negative size
        assert _raw_decode(lib, d) == 1
    d = descs()
    d[2].stride[2] = 256                                      # (bs, D) tile not contiguous
    assert _raw_decode(lib, d) == 1 and b"tile" in lib.pkv_last_error()
    d = descs()
    d[1].stride[2] = 2                                        # query's last dim strided
    assert _raw_decode(lib, d) == 1 and b"contiguous" in lib.pkv_last_error()
    d = descs()
    d[4].dtype = 4                                            # int64 block table: known, unsupported
    assert _raw_decode(lib, d) == 2


def test_window_prefill_and_noalloc_validation(dry):
    a = _decode_args()
    assert _status(binding.paged_attention_decode, **a, sliding_window=64) == 0
    assert _status(binding.paged_attention_decode, **a, sliding_window=-1) == 1
    assert _status(binding.paged_attention_decode_noalloc, **a) == 0
    b = dict(a)
    b["num_kv_heads"] = 3
    assert _status(binding.paged_attention_decode_noalloc, **b) == 1
    # prefill: 5 packed new tokens of 3 sequences
    T = 5
    q = torch.zeros(T, 8, 128, dtype=torch.bfloat16)
    p = dict(out=torch.empty_like(q), query=q, key_cache=a["key_cache"], value_cache=a["value_cache"],
             block_tables=a["block_tables"], context_lens=torch.full((3,), 8, dtype=torch.int32),
             query_start_loc=torch.tensor([0, 2, 4, 5], dtype=torch.int32), num_kv_heads=2, scale=0.1,
             block_size=16, max_blocks_per_seq=4)
    # the prefill kernel needs the driver's tensor-map encoder: without a GPU driver a
    # valid call passes every argument check and then reports UNSUPPORTED
    assert _status(binding.paged_attention_prefill, **p) in ((0,) if torch.cuda.is_available() else (0, 2))
    assert _status(binding.paged_attention_prefill, **dict(p, query_start_loc=torch.tensor([0, 2, 5], dtype=torch.int32))) == 1
    f = torch.zeros(T, 8, 128, dtype=torch.float32)
    assert _status(binding.paged_attention_prefill, **dict(p, query=f, out=torch.empty_like(f))) == 2


def test_workspace_errors_and_empty_pool(dry):
    lib = binding.load_library()
    assert lib.pkv_reserve_workspace(ctypes.c_int64(-1)) == 1
    assert lib.pkv_read_device_errors(None) == 1 and b"null" in lib.pkv_last_error()
    a = _decode_args(NB=0)                                   # a pool of no blocks
    assert _status(binding.paged_attention_decode, **a) == 1 and b"no block" in lib.pkv_last_error()


def test_last_error_is_per_thread(dry):
    """pkv_last_error() is the calling thread's message: another thread's failure does
    not replace it."""
    import threading
    lib = binding.load_library()
    a = _decode_args()
    a["num_kv_heads"] = 3
    with pytest.raises(binding.PkvError):
        binding.paged_attention_decode(**a)
    mine = lib.pkv_last_error()
    assert b"num_kv_heads" in mine
    theirs = []

    def other():
        b = _decode_args()
        b["scale"] = float("nan")
        try:
            binding.paged_attention_decode(**b)
        except binding.PkvError:
            pass
        theirs.append(lib.pkv_last_error())
    t = threading.Thread(target=other)
    t.start()
    t.join()
    assert b"scale" in theirs[0]
    assert lib.pkv_last_error() == mine


def test_call_descriptors_are_cached_by_content(lib):
    """The wrappers' descriptor cache hands out a descriptor equal to a fresh one, keyed
    by everything a descriptor holds: another view, dtype, scale or per-head scale array
    gets its own; empty tensors carry no pointer; the cache stays bounded."""
    def fields(d):
        return (d.data, d.dtype, d.ndim, tuple(d.shape), tuple(d.stride), d.scale, d.head_scales)

    binding._DESC_CACHE.clear()
    c = torch.zeros(6, 2, 16, 64, dtype=torch.bfloat16)
    hs = torch.ones(2, dtype=torch.float32)
    for t, sc, h in ((c, 1.0, None), (c[1:], 1.0, None), (c.view(torch.float8_e4m3fn)[:, :1], 1.0, None),
                     (c, 0.5, None), (c.view(torch.float8_e4m3fn)[..., :64], 0.5, hs), (c[:0], 1.0, None)):
        r = binding._ref(t, sc, h)
        assert binding._ref(t, sc, h) is r                         # a hit
        assert fields(r._obj) == fields(binding.describe(t, sc, h))
    assert len(binding._DESC_CACHE) == 6
    assert binding._ref(c[:0])._obj.data is None
    for i in range(binding._DESC_CACHE_MAX + 10):
        binding._ref(c, float(i))
    assert len(binding._DESC_CACHE) <= binding._DESC_CACHE_MAX


def test_zero_heads_queue_nothing(lib):
    """A batch with no query head (decode, prefill) or a pool with no KV head (write,
    copy) has nothing to compute: the call returns OK before it touches a device (so it
    succeeds here, where there is none), rather than launching kernels whose tile
    counts would be zero."""
    binding.set_option("dry_run", 0)
    a = _decode_args(Hq=0)
    assert _status(binding.paged_attention_decode, **a) == 0
    assert _status(binding.paged_attention_decode, **a, sliding_window=16) == 0
    q = torch.zeros(5, 0, 128, dtype=torch.bfloat16)
    assert _status(binding.paged_attention_prefill, out=torch.empty_like(q), query=q, key_cache=a["key_cache"],
                   value_cache=a["value_cache"], block_tables=a["block_tables"],
                   context_lens=torch.full((3,), 8, dtype=torch.int32),
                   query_start_loc=torch.tensor([0, 2, 4, 5], dtype=torch.int32), num_kv_heads=2, scale=0.1,
                   block_size=16, max_blocks_per_seq=4) in ((0,) if torch.cuda.is_available() else (0, 2))
    c0 = torch.zeros(10, 0, 16, 128, dtype=torch.bfloat16)
    k0 = torch.zeros(4, 0, 128, dtype=torch.bfloat16)
    assert _status(binding.reshape_and_cache, key=k0, value=k0, key_cache=c0, value_cache=c0,
                   slot_mapping=torch.arange(4, dtype=torch.int64)) == 0
    assert _status(binding.copy_blocks, cache=c0, src_dst_pairs=torch.tensor([[0, 1]], dtype=torch.int64)) == 0
