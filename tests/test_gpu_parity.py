"""GPU parity: the CUDA path through the C ABI against the CPU oracle, on the same
seeded inputs.  Cache writes and block copies must match bit for bit; decode outputs
within the stated max-abs tolerances (f32 1e-5, bf16 2e-2, fp8 K/V 5e-2) and, more
tightly, within the final output rounding (2^-8 relative for a bf16 output)."""
import os

import pytest
import numpy as np
import torch

import oracle
from paged_kv_cache_90_gb300 import binding
from paged_kv_cache_90_gb300 import build as pkv_build
from paged_kv_cache_90_gb300 import workloads as wl
from paged_kv_cache_90_gb300.decode_step import DeviceWorkload, prepare_step

pytestmark = pytest.mark.gpu

THREADS = max(1, min(16, len(os.sched_getaffinity(0))))
MAX_ABS = {torch.float32: 1e-5, torch.bfloat16: 2e-2, torch.float8_e4m3fn: 5e-2}


@pytest.fixture(scope="module", autouse=True)
def _setup():
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    pkv_build.build()
    oracle.build()
    binding.load_library()
    yield
    binding.set_option("partition_tokens", 0)
    binding.set_option("debug_sync", 0)


@pytest.fixture(params=["tensor", "core"])
def kernel(request):
    """Run the test with the tensor-core kernel forced, then with the CUDA-core one."""
    binding.set_option("decode_kernel", 2 if request.param == "tensor" else 1)
    yield request.param
    binding.set_option("decode_kernel", 0)


@pytest.fixture(params=["tcgen05", "mma_sync"])
def pkernel(request):
    """Run a prefill test on the tcgen05 kernel (accumulators in tensor memory), then on
    the mma.sync one."""
    binding.set_option("prefill_kernel", 2 if request.param == "tcgen05" else 1)
    yield request.param
    binding.set_option("prefill_kernel", 0)


@pytest.fixture
def partition_tokens():
    def set_(n):
        binding.set_option("partition_tokens", n)
    yield set_
    binding.set_option("partition_tokens", 0)


def run_device(w):
    dw = DeviceWorkload(w)
    outs = []
    for i in range(len(w.steps)):
        outs.append(dw.run_step(i, out=torch.empty_like(dw.out)).clone())
    torch.cuda.synchronize()
    assert binding.read_device_errors() == 0
    return [o.double().cpu() for o in outs], dw.key_cache.cpu(), dw.value_cache.cpu()


def run_oracle(w):
    kc, vc = w.key_cache.clone(), w.value_cache.clone()
    outs = [oracle.run_workload_step(w, i, kc, vc, THREADS) for i in range(len(w.steps))]
    return outs, kc, vc


def raw(t):
    return t.view(torch.uint8) if t.element_size() == 1 else t.view(torch.int16 if t.element_size() == 2 else torch.int32)


def gather_blocks(cache, blocks):
    if cache.dtype == torch.float8_e4m3fn:   # torch cannot index fp8 tensors on the CPU
        return cache.view(torch.uint8)[blocks].view(torch.float8_e4m3fn)
    return cache[blocks]


def weighted_abs_values(w, st, kc, vc):
    """sum_j p_j |V_j| for every output (softmax weights p), in fp64 with torch on the
    gathered context: the scale of the error that rounding the weights to a 16-bit
    format before the P.V product can cause (at most 2^-9 of it for bf16)."""
    S, hq, d = st.query.shape
    hk, bs = w.num_kv_heads, w.block_size
    g = hq // hk
    W = w.sliding_window
    out = torch.zeros(S, hq, d, dtype=torch.float64)
    for s in range(S):
        L = int(st.context_lens[s])
        if L == 0:
            continue
        lo = max(0, L - W) if W > 0 else 0       # first attended position
        b0 = lo // bs                            # blocks before it may be released (-1)
        n = -(-L // bs) - b0
        blocks = st.block_tables[s, b0:b0 + n].long()
        K = gather_blocks(kc, blocks).double().permute(1, 0, 2, 3).reshape(hk, n * bs, d)[:, lo - b0 * bs:L - b0 * bs]
        V = gather_blocks(vc, blocks).double().permute(1, 0, 2, 3).reshape(hk, n * bs, d)[:, lo - b0 * bs:L - b0 * bs]
        ks = w.k_head_scales.double().view(hk, 1, 1) if w.k_head_scales is not None else w.k_scale
        vs = w.v_head_scales.double().view(hk, 1, 1) if w.v_head_scales is not None else w.v_scale
        K = K * ks
        V = V.abs() * vs
        q = st.query[s].double().view(hk, g, d)
        p = torch.softmax(w.scale * q @ K.transpose(1, 2), dim=-1)
        out[s] = (p @ V).reshape(hq, d)
    return out


def weighted_abs_values_prefill(w, st, kc, vc):
    """sum_j p_j |V_j| for every packed query row of a prefill step (causal softmax over
    positions 0..p), in fp64 with torch."""
    T, hq, d = st.query.shape
    hk, bs = w.num_kv_heads, w.block_size
    g = hq // hk
    out = torch.zeros(T, hq, d, dtype=torch.float64)
    qsl = st.query_start_loc.tolist()
    for s in range(len(qsl) - 1):
        L, n = int(st.context_lens[s]), qsl[s + 1] - qsl[s]
        if n == 0:
            continue
        nb = -(-L // bs)
        blocks = st.block_tables[s, :nb].long()
        K = gather_blocks(kc, blocks).double().permute(1, 0, 2, 3).reshape(hk, nb * bs, d)[:, :L]
        V = gather_blocks(vc, blocks).double().permute(1, 0, 2, 3).reshape(hk, nb * bs, d)[:, :L].abs()
        q = st.query[qsl[s]:qsl[s + 1]].double().view(n, hk, g, d).permute(1, 2, 0, 3)   # [hk, g, n, d]
        z = w.scale * q @ K.transpose(1, 2)[:, None]                                      # [hk, g, n, L]
        mask = torch.arange(L)[None, :] > (L - n + torch.arange(n))[:, None]
        p = torch.softmax(z.masked_fill(mask, float("-inf")), dim=-1)
        out[qsl[s]:qsl[s + 1]] = (p @ V[:, None]).permute(2, 0, 1, 3).reshape(n, hq, d)
    return out


def assert_decode_close(got, ref, w, wabs=None):
    err = (got - ref).abs()
    assert torch.isfinite(got).all()
    worst = MAX_ABS[w.kv_dtype] if w.kv_dtype == torch.float8_e4m3fn else MAX_ABS[w.q_dtype]
    assert err.max().item() <= worst, f"max abs err {err.max().item()} > {worst}"
    # rounding bound: the output's own rounding plus (tensor-core path) the 16-bit
    # weights of the P.V product, with a factor-2 margin
    if w.q_dtype == torch.bfloat16:
        tight = 2.0 ** -8 * ref.abs() + 2e-5
    else:
        tight = 2e-6 * ref.abs() + 2e-6
    if wabs is not None:
        tight = tight + 2.0 ** -8 * wabs
    bad = (err > tight).sum().item()
    assert bad == 0, f"{bad} outputs beyond the rounding bound (max err {err.max().item():.3e})"


def check_workload(w):
    outs, kc, vc = run_device(w)
    kc0, vc0 = w.key_cache.clone(), w.value_cache.clone()
    routs, wabs = [], []
    for i in range(len(w.steps)):
        routs.append(oracle.run_workload_step(w, i, kc0, vc0, THREADS))
        wa = None
        if w.q_dtype == torch.bfloat16:
            wa = (weighted_abs_values_prefill if w.steps[i].query_start_loc is not None
                  else weighted_abs_values)(w, w.steps[i], kc0, vc0)
        wabs.append(wa)
    assert torch.equal(raw(kc), raw(kc0)), "key cache differs from the oracle's"
    assert torch.equal(raw(vc), raw(vc0)), "value cache differs from the oracle's"
    for got, ref, wa in zip(outs, routs, wabs):
        assert_decode_close(got, ref, w, wa)
    return outs, routs


# --- the five workloads, scaled to seconds of oracle time and at full size ----------

def test_tiny_f32():
    check_workload(wl.tiny())


@pytest.mark.parametrize("layout", [(0, 1), (4, 1), (5, 2)])
def test_scalar_example_padded(layout):
    """keys 0, query 1, values 1..5 at block size 4: 3 for every layout (head padded
    with zeros to 64 dims, which leaves q.k unchanged)."""
    w = wl.scalar_example(physical=layout, num_blocks=8, head_dim=64)
    outs, _, _ = run_device(w)
    got = outs[0][0, 0]
    assert abs(got[0].item() - 3.0) <= 1e-6
    assert torch.all(got[1:] == 0)


@pytest.mark.parametrize("bs", [8, 16, 32])
def test_llama3_shaped_small(bs, kernel):
    check_workload(wl.llama3_8b_decode(seed=2, num_seqs=8, len_range=(128, 600), block_size=bs, poison=True))


def test_llama3_shaped_peaked_queries(kernel):
    """Queries scaled by 8: concentrated attention, |out| of order 1."""
    w = wl.llama3_8b_decode(seed=21, num_seqs=6, len_range=(100, 900), poison=True)
    w.steps[0].query.mul_(8)
    outs, routs = check_workload(w)
    assert routs[0].abs().max() > 0.5


def test_llama3_shaped_full(kernel):
    check_workload(wl.llama3_8b_decode())


@pytest.mark.parametrize("bs", [16, 32])
def test_long_context_small(bs, kernel):
    check_workload(wl.long_context(block_size=bs, num_seqs=2, context_len=5000, poison=True))


@pytest.mark.parametrize("bs", [16, 32])
def test_long_context_full(bs, kernel):
    check_workload(wl.long_context(block_size=bs))


def test_shared_prefix_cow_small(kernel):
    w = wl.shared_prefix_cow(num_groups=4, prefix_blocks=8, suffix_range=(16, 120), poison=True)
    assert w.steps[0].cow_pairs.shape[0] == 12
    check_workload(w)


def test_shared_prefix_cow_full(kernel):
    w = wl.shared_prefix_cow()
    assert w.steps[0].cow_pairs.shape[0] == 96
    check_workload(w)


@pytest.mark.parametrize("kv", ["bf16", "e4m3"])
@pytest.mark.parametrize("bs", [8, 16, 32])
def test_continuous_batching_small(bs, kv, kernel):
    check_workload(wl.continuous_batching(block_size=bs, kv_dtype=kv, num_seqs=24, num_steps=3,
                                          median=200, cap=2000, poison=True))


@pytest.mark.parametrize("kv", ["bf16", "e4m3"])
@pytest.mark.parametrize("bs", [8, 16, 32])
def test_continuous_batching_full(bs, kv, kernel):
    check_workload(wl.continuous_batching(block_size=bs, kv_dtype=kv))


# --- prefill / chunked prefill ----------------------------------------------------

@pytest.mark.parametrize("bs", [8, 16, 32])
@pytest.mark.parametrize("heads", [(32, 8), (16, 16), (16, 8), (32, 2), (12, 4)])
def test_prefill_small(bs, heads, pkernel):
    """Prompts and later chunks of different lengths (tile edges, prefixes off the
    stage grid), GQA groups 1 to 16, every unused slot NaN."""
    hq, hk = heads
    check_workload(wl.chunked_prefill(seed=90 + bs + hq + hk, prefix_lens=(0, 0, 5, 37, 16, 200, 0),
                                      chunk_lens=(1, 17, 33, 64, 127, 40, 130), num_heads=hq, num_kv_heads=hk,
                                      head_dim=128 if hq != 12 else 64, block_size=bs, poison=True))


def test_prefill_empty_chunk_and_single_tokens(pkernel):
    """A sequence with no new token leaves nothing to write; one-token chunks equal
    decode (checked against the oracle like every prefill)."""
    check_workload(wl.chunked_prefill(seed=95, prefix_lens=(10, 300, 0, 47), chunk_lens=(1, 1, 1, 1), poison=True))
    w = wl.chunked_prefill(seed=96, prefix_lens=(10, 20, 30), chunk_lens=(5, 1, 9), poison=True)
    st = w.steps[0]
    # drop the middle sequence's chunk: its context shrinks to its prefix, no rows
    keep = torch.tensor([0, 1, 2, 3, 4, 6, 7, 8, 9, 10, 11, 12, 13, 14])
    st.query, st.new_key, st.new_value = st.query[keep], st.new_key[keep], st.new_value[keep]
    st.slot_mapping = st.slot_mapping[keep]
    st.context_lens = torch.tensor([15, 20, 39], dtype=torch.int32)
    st.query_start_loc = torch.tensor([0, 5, 5, 14], dtype=torch.int32)
    check_workload(w)


@pytest.mark.parametrize("num_seqs", [40, 70])
def test_prefill_many_sequences(num_seqs, pkernel):
    """Many sequences, prefix and chunk lengths repeating (so that tile pairs see equal
    key counts): up to 64 sequences the tcgen05 kernel takes the pairs in decreasing
    key count, equal counts by sequence, beyond 64 sequence by sequence; either way
    every pair is computed once (unused slots NaN)."""
    prefix = tuple((i % 5) * 60 for i in range(num_seqs))
    chunks = tuple(1 + (i % 7) * 30 for i in range(num_seqs))
    check_workload(wl.chunked_prefill(seed=97 + num_seqs, prefix_lens=prefix, chunk_lens=chunks, poison=True))


def test_prefill_full(pkernel):
    """Llama-3-8B-shaped prefill: two 2048-token prompts and two 512-token chunks of
    long prompts (prefixes 512 and 1536)."""
    check_workload(wl.chunked_prefill())


@pytest.mark.parametrize("bs", [8, 16, 32])
def test_fp8_head_scales_small(bs, kernel):
    """An 8-bit cache whose KV heads differ by 2^3 in magnitude, one scale per head:
    the write quantises each head with its scale and decode dequantises with it."""
    check_workload(wl.continuous_batching(seed=70 + bs, block_size=bs, kv_dtype="e4m3", num_seqs=24, num_steps=3,
                                          median=200, cap=2000, poison=True, head_spread=3.0))


def test_fp8_head_scales_full(kernel):
    check_workload(wl.continuous_batching(kv_dtype="e4m3", head_spread=3.0))


@pytest.mark.parametrize("kv", ["bf16", "e4m3", "f32"])
def test_write_reports_amax(kv):
    """The amax report equals the oracle's per-head max |x| (bf16 / f32 sources are
    exact in fp32), keeps a larger starting value, skips padding tokens, and turns NaN
    for a head whose source holds a NaN."""
    dt = "f32" if kv == "f32" else "bf16"
    w = wl.variable_length_decode("a", 73, [5, 40, 99, 7], 8, 4, 128, 16, kv, q_dtype=dt, num_steps=1,
                                  head_spread=4.0 if kv == "e4m3" else 0.0)
    st = w.steps[0]
    dw = DeviceWorkload(w)
    sm = st.slot_mapping.clone()
    sm[2] = -1
    key, value = st.new_key.clone(), st.new_value.clone()
    key[1, 3, 17] = float("nan")
    ka = torch.zeros(4, dtype=torch.float32, device="cuda")
    va = torch.full((4,), 1e9, dtype=torch.float32, device="cuda")
    binding.reshape_and_cache(key.cuda(), value.cuda(), dw.key_cache, dw.value_cache, sm.cuda(), w.k_scale,
                              w.v_scale, None, dw.k_head_scales, dw.v_head_scales, ka, va)
    torch.cuda.synchronize()
    ref_k = torch.zeros(4, dtype=torch.float64)
    ref_v = torch.zeros(4, dtype=torch.float64)
    kc, vc = w.key_cache.clone(), w.value_cache.clone()
    oracle.reshape_and_cache(key, value, kc, vc, sm, w.k_scale, w.v_scale, w.k_head_scales, w.v_head_scales,
                             ref_k, ref_v)
    got_k = ka.cpu().double()
    assert torch.isnan(got_k[3]) and torch.isnan(ref_k[3])
    assert torch.equal(got_k[:3], ref_k[:3])
    assert torch.equal(va.cpu(), torch.full((4,), 1e9))
    assert torch.equal(raw(dw.key_cache.cpu()), raw(kc)) and torch.equal(raw(dw.value_cache.cpu()), raw(vc))
    assert binding.read_device_errors() == 0


@pytest.mark.parametrize("bs", [8, 16, 32])
@pytest.mark.parametrize("window", [1, 7, 16, 17, 100])
def test_sliding_window_small(bs, window, kernel):
    """Windows shorter than, around and beyond a stage / block; blocks before each
    window released (table entries -1, slots NaN) and handed out again."""
    check_workload(wl.sliding_window_decode(seed=60 + window + bs, num_seqs=12, window=window, block_size=bs,
                                            num_steps=2, len_range=(1, 600), poison=True))


@pytest.mark.parametrize("kv", ["bf16", "e4m3"])
def test_sliding_window_full(kv, kernel):
    """8 sequences of 32768 tokens, window 4096 (the benchmark's sliding-window layer)."""
    check_workload(wl.sliding_window_decode(kv_dtype=kv))


@pytest.mark.parametrize("kv", ["bf16", "e4m3"])
def test_fused_append_writes_only_where_told(kv):
    """A token with slot -1 writes nothing; a token whose slot is not its sequence's
    newest position is stored there (the decode then reads the cache as it was), exactly
    as the write-then-decode calls do."""
    w = wl.llama3_8b_decode(seed=62, num_seqs=6, len_range=(20, 300), kv_dtype=kv)
    st = w.steps[0]
    st.slot_mapping = st.slot_mapping.clone()
    st.slot_mapping[1] = -1
    # sequence 3's token goes to an unused slot (never read in this step)
    used = set()
    for r, L in zip(st.block_tables.tolist(), st.context_lens.tolist()):
        for p in range(L):
            used.add(r[p // w.block_size] * w.block_size + p % w.block_size)
    st.slot_mapping[3] = next(x for x in range(w.num_blocks * w.block_size) if x not in used)
    runs = {}
    for joint in ("fused", False):
        dw = DeviceWorkload(w)
        binding.set_option("fused_append", 2)   # the write inside the kernel for both cache types
        try:
            o = dw.run_step(0, out=torch.empty_like(dw.out), joint=joint).clone()
        finally:
            binding.set_option("fused_append", 0)
        torch.cuda.synchronize()
        runs[joint] = (o, dw.key_cache.clone(), dw.value_cache.clone())
    assert binding.read_device_errors() == 0
    assert torch.equal(runs["fused"][0], runs[False][0])
    assert torch.equal(raw(runs["fused"][1]), raw(runs[False][1]))
    assert torch.equal(raw(runs["fused"][2]), raw(runs[False][2]))


def test_window_covering_every_context_is_the_plain_decode(kernel):
    """A window no shorter than any context gives the plain decode's bits."""
    w = wl.llama3_8b_decode(seed=61, num_seqs=8, len_range=(1, 900))
    dw = DeviceWorkload(w)
    dw.run_step(0)
    st = dw.steps[0]
    args = (st.query, dw.key_cache, dw.value_cache, st.block_tables, st.context_lens, w.num_kv_heads, w.scale,
            w.block_size, w.max_blocks_per_seq)
    plain = binding.paged_attention_decode(torch.empty_like(dw.out), *args).clone()
    for window in (901, 5000):
        got = binding.paged_attention_decode(torch.empty_like(dw.out), *args, sliding_window=window)
        torch.cuda.synchronize()
        assert torch.equal(got, plain)
    assert binding.read_device_errors() == 0


# --- edge cases -----------------------------------------------------------------

def test_partition_edges(partition_tokens, kernel):
    """Lengths around partition and block boundaries with 256-token partitions, so the
    log-sum-exp reduce merges 1..5 partitions."""
    partition_tokens(256)
    check_workload(wl.variable_length_decode("edges", 30, [1, 2, 255, 256, 257, 511, 512, 513, 1000, 1280],
                                             8, 2, 128, 16, "bf16", poison=True))


@pytest.mark.parametrize("hq,hk,d,bs,kv,q", [
    (6, 2, 128, 16, "bf16", "bf16"),    # 3 query heads per KV head -> one head per block
    (16, 2, 128, 16, "bf16", "bf16"),   # 8 per KV head
    (32, 2, 128, 16, "bf16", "bf16"),   # 16 per KV head: both MMA row halves hold heads
    (16, 1, 64, 8, "bf16", "bf16"),     # 16 per KV head, head_dim 64
    (32, 2, 128, 32, "e4m3", "bf16"),   # 16 per KV head, 8-bit cache
    (4, 4, 128, 16, "bf16", "bf16"),    # no grouping
    (8, 2, 64, 2, "bf16", "bf16"),      # head_dim 64, block size 2
    (8, 4, 64, 4, "e4m3", "bf16"),
    (8, 2, 128, 8, "bf16", "f32"),      # f32 queries over a bf16 cache
    (4, 2, 128, 32, "f32", "f32"),
    (16, 2, 64, 8, "e4m3", "f32"),
])
def test_shapes_and_dtypes(hq, hk, d, bs, kv, q):
    check_workload(wl.variable_length_decode("shapes", 40 + hq + d + bs, [1, 7, bs, 3 * bs + 1, 300, 777],
                                             hq, hk, d, bs, kv, q_dtype=q, poison=True, num_steps=2))


def test_zero_length_and_empty_batch():
    w = wl.variable_length_decode("z", 50, [5, 40], 8, 2, 128, 16, "bf16", poison=True)
    dw = DeviceWorkload(w)
    st = dw.steps[0]
    dw.run_step(0)
    cl = st.context_lens.clone()
    cl[0] = 0
    out = torch.full_like(dw.out, 7.0)
    binding.paged_attention_decode(out, st.query, dw.key_cache, dw.value_cache, st.block_tables, cl,
                                   w.num_kv_heads, w.scale, w.block_size, w.max_blocks_per_seq)
    torch.cuda.synchronize()
    assert torch.all(out[0] == 0)
    # an empty batch is a no-op
    e = torch.empty(0, 8, 128, dtype=torch.bfloat16, device="cuda")
    binding.paged_attention_decode(e, e, dw.key_cache, dw.value_cache,
                                   torch.empty(0, w.max_blocks_per_seq, dtype=torch.int32, device="cuda"),
                                   torch.empty(0, dtype=torch.int32, device="cuda"),
                                   w.num_kv_heads, w.scale, w.block_size, w.max_blocks_per_seq)
    assert binding.read_device_errors() == 0


def test_strided_cache_views_and_side_stream():
    """K and V as views of one [NB, 2, Hk, bs, D] tensor, work on a non-default stream."""
    w = wl.variable_length_decode("views", 60, [3, 90, 400], 8, 2, 128, 16, "bf16", poison=True)
    nb = w.num_blocks
    both = torch.empty(nb, 2, 2, 16, 128, dtype=torch.bfloat16, device="cuda")
    both[:, 0] = w.key_cache.cuda()
    both[:, 1] = w.value_cache.cuda()
    kc, vc = both[:, 0], both[:, 1]
    st = DeviceWorkload(w).steps[0]
    out = torch.empty(3, 8, 128, dtype=torch.bfloat16, device="cuda")
    s = torch.cuda.Stream()
    s.wait_stream(torch.cuda.current_stream())
    with torch.cuda.stream(s):
        binding.reshape_and_cache(st.new_key, st.new_value, kc, vc, st.slot_mapping)
        binding.paged_attention_decode(out, st.query, kc, vc, st.block_tables, st.context_lens, 2, w.scale,
                                       16, w.max_blocks_per_seq)
        pairs = torch.tensor([[int(st.block_tables[0, 0]), nb - 1]], dtype=torch.int64, device="cuda")
    s.synchronize()
    routs, rkc, rvc = run_oracle(w)
    assert_decode_close(out.double().cpu(), routs[0], w, weighted_abs_values(w, w.steps[0], rkc, rvc))
    assert torch.equal(raw(kc.cpu()), raw(rkc))
    with torch.cuda.stream(s):
        binding.copy_blocks(kc, pairs)
    s.synchronize()
    assert torch.equal(raw(kc[nb - 1].cpu()), raw(rkc[int(st.block_tables[0, 0])]))
    assert torch.equal(raw(vc.cpu()), raw(rvc))       # V untouched by the K copy


@pytest.mark.parametrize("src,dst", [("f32", "f32"), ("bf16", "bf16"), ("bf16", "e4m3"), ("f32", "e4m3")])
def test_cache_write_bit_exact(src, dst):
    """Every slot kind: regular, padding (-1), first/last slot of the pool; e4m3 with
    values beyond the saturation point."""
    g = torch.Generator().manual_seed(70)
    nb, hk, bs, d, t = 12, 4, 16, 128, 40
    dt = wl.DTYPES
    kc = torch.randn(nb, hk, bs, d, generator=g).to(dt[dst] if dst != "e4m3" else torch.float32)
    if dst == "e4m3":
        kc = (kc / 0.02).clamp(-448, 448).to(torch.float8_e4m3fn)
    vc = kc.clone()
    key = (torch.randn(t, hk, d, generator=g) * 3).to(dt[src])
    value = (torch.randn(t, hk, d, generator=g) * 50).to(dt[src])
    slots = torch.randperm(nb * bs, generator=g)[:t]
    slots[3] = -1
    slots[7] = 0
    slots[8] = nb * bs - 1
    ks, vs = (0.02, 0.05) if dst == "e4m3" else (1.0, 1.0)
    dk, dv = kc.cuda(), vc.cuda()
    binding.reshape_and_cache(key.cuda(), value.cuda(), dk, dv, slots.cuda(), ks, vs)
    torch.cuda.synchronize()
    rk, rv = kc.clone(), vc.clone()
    oracle.reshape_and_cache(key, value, rk, rv, slots, ks, vs)
    assert torch.equal(raw(dk.cpu()), raw(rk))
    assert torch.equal(raw(dv.cpu()), raw(rv))
    assert binding.read_device_errors() == 0


def _e4m3_boundary_values(scale: float, n: int, g) -> torch.Tensor:
    """n binary32 values x whose quotients x / scale sit on, next to and between the
    rounding midpoints of the e4m3 codes (both signs), plus zeros, infinities, values
    past saturation, tiny and huge magnitudes, and random ones."""
    mags = oracle.e4m3_decode(np.arange(0x7F, dtype=np.uint8)).tolist()   # 0 .. 448
    q = []
    for a, b in zip(mags, mags[1:]):
        mid = np.float32((a + b) / 2)
        q += [mid, np.nextafter(mid, np.float32(np.inf)), np.nextafter(mid, np.float32(0))]
    q = np.array(q, dtype=np.float64)
    x = np.concatenate([q * scale, -q * scale]).astype(np.float32)   # quotient ~ midpoint after rounding x
    special = np.array([0.0, -0.0, np.inf, -np.inf, 449.0 * scale, -1e4 * scale, 2.0 ** -110, -(2.0 ** 101),
                        1e-30, 3e38], dtype=np.float32)
    rnd = (torch.randn(n, generator=g, dtype=torch.float64) * 100 * scale).numpy().astype(np.float32)
    return torch.from_numpy(np.concatenate([x, special, rnd])[:n].copy())


@pytest.mark.parametrize("path", ["write", "fused"])
def test_e4m3_encode_rounding_boundaries(path):
    """The 8-bit encode (x / scale in binary32, then the nearest e4m3 code) is bit exact
    where the quotient sits on or next to a rounding midpoint, for scales inside and
    outside the reciprocal-based division's range, in the cache write and in the fused
    append."""
    g = torch.Generator().manual_seed(71)
    scales = [0.02, 1 / 3, 0.0173, 1.0, 7.3, 1e-7, 3e6, 2.0 ** -20]
    hk, d, S = len(scales), 128, 8
    w = wl.variable_length_decode("rounding", 72, [33, 17, 64, 5, 48, 16, 90, 2], 4 * hk, hk, d, 16, "e4m3",
                                  head_spread=1.0)
    st = w.steps[0]
    w.k_head_scales = torch.tensor(scales, dtype=torch.float32)
    w.v_head_scales = torch.tensor(scales[::-1], dtype=torch.float32)
    key = torch.stack([_e4m3_boundary_values(sc, S * d, g).view(S, d) for sc in scales], dim=1)
    value = torch.stack([_e4m3_boundary_values(sc, S * d, g).view(S, d) for sc in scales[::-1]], dim=1)
    perm = torch.randperm(S * d, generator=g)                        # mix the lanes that see each case
    key = key.permute(0, 2, 1).reshape(S * d, hk)[perm].reshape(S, d, hk).permute(0, 2, 1).contiguous()
    st.new_key, st.new_value = key, value.contiguous()
    rk, rv = w.key_cache.clone(), w.value_cache.clone()
    oracle.reshape_and_cache(key, st.new_value, rk, rv, st.slot_mapping, k_head_scales=w.k_head_scales,
                             v_head_scales=w.v_head_scales)
    dw = DeviceWorkload(w)
    dst = dw.steps[0]
    if path == "write":
        binding.reshape_and_cache(dst.new_key, dst.new_value, dw.key_cache, dw.value_cache, dst.slot_mapping,
                                  k_head_scales=dw.k_head_scales, v_head_scales=dw.v_head_scales)
    else:
        binding.set_option("decode_kernel", 2)
        binding.set_option("fused_append", 2)
        try:
            dw.run_step(0, joint="fused")
        finally:
            binding.set_option("decode_kernel", 0)
            binding.set_option("fused_append", 0)
    torch.cuda.synchronize()
    assert binding.read_device_errors() == 0
    assert torch.equal(raw(dw.key_cache.cpu()), raw(rk))
    assert torch.equal(raw(dw.value_cache.cpu()), raw(rv))


def test_copy_blocks_bit_exact():
    g = torch.Generator().manual_seed(80)
    cache = torch.randn(40, 8, 16, 128, generator=g).to(torch.bfloat16)
    pairs = torch.tensor([[1, 30], [5, 31], [5, 32], [39, 0], [17, 18]], dtype=torch.int64)
    d = cache.cuda()
    binding.copy_blocks(d, pairs.cuda())
    torch.cuda.synchronize()
    ref = cache.clone()
    oracle.copy_blocks(ref, pairs)
    assert torch.equal(raw(d.cpu()), raw(ref))


def test_device_checks_flag_bad_indices():
    """Out-of-range table entries, slots, copy pairs and context lengths are caught
    on the device: the access is skipped or redirected in bounds and a bit is set."""
    w = wl.variable_length_decode("bad", 90, [20, 40], 8, 2, 128, 16, "bf16")
    dw = DeviceWorkload(w)
    st = dw.steps[0]
    assert binding.read_device_errors() == 0
    bt = st.block_tables.clone()
    bt[1, 1] = w.num_blocks + 3
    binding.paged_attention_decode(dw.out, st.query, dw.key_cache, dw.value_cache, bt, st.context_lens,
                                   2, w.scale, 16, w.max_blocks_per_seq)
    assert binding.read_device_errors() == binding.DEVERR["table_entry"]
    sm = st.slot_mapping.clone()
    sm[0] = w.num_blocks * 16
    before = dw.key_cache.clone()
    binding.reshape_and_cache(st.new_key[:1], st.new_value[:1], dw.key_cache, dw.value_cache, sm[:1])
    assert binding.read_device_errors() == binding.DEVERR["slot"]
    assert torch.equal(raw(dw.key_cache), raw(before))
    binding.copy_blocks(dw.key_cache, torch.tensor([[0, w.num_blocks]], dtype=torch.int64, device="cuda"))
    assert binding.read_device_errors() == binding.DEVERR["copy_pair"]
    cl = st.context_lens.clone()
    cl[0] = w.max_blocks_per_seq * 16 + 1
    binding.paged_attention_decode(dw.out, st.query, dw.key_cache, dw.value_cache, st.block_tables, cl,
                                   2, w.scale, 16, w.max_blocks_per_seq)
    assert binding.read_device_errors() & binding.DEVERR["context_len"]
    binding.set_option("debug_sync", 1)
    try:
        with pytest.raises(binding.PkvError) as ei:
            binding.paged_attention_decode(dw.out, st.query, dw.key_cache, dw.value_cache, bt,
                                           st.context_lens, 2, w.scale, 16, w.max_blocks_per_seq)
        assert ei.value.status == 4
    finally:
        binding.set_option("debug_sync", 0)
    assert binding.read_device_errors() == 0


def test_copy_blocks_overlap_check_under_debug_sync():
    """With debug sync on, copy pairs that break the parallel copy's precondition (a
    destination named twice, or a destination that is also a source) are reported as a
    device-check failure with the overlap bit; valid pairs still copy bit for bit, and
    with debug sync off no check runs."""
    g = torch.Generator().manual_seed(81)
    cache = torch.randn(24, 4, 16, 64, generator=g).to(torch.bfloat16)
    d = cache.cuda()
    assert binding.read_device_errors() == 0
    binding.set_option("debug_sync", 1)
    try:
        for bad in ([[1, 5], [2, 5]], [[1, 2], [2, 3]], [[3, 3]], [[0, 9], [4, 10], [9, 11]]):
            with pytest.raises(binding.PkvError) as ei:
                binding.copy_blocks(d, torch.tensor(bad, dtype=torch.int64, device="cuda"))
            assert ei.value.status == 4 and "0x20" in ei.value.message, ei.value.message
        assert binding.read_device_errors() == 0          # the failing call cleared the word
        good = torch.tensor([[1, 12], [2, 13], [1, 14], [23, 0]], dtype=torch.int64)
        d = cache.cuda()
        binding.copy_blocks(d, good.cuda())
        ref = cache.clone()
        oracle.copy_blocks(ref, good)
        assert torch.equal(raw(d.cpu()), raw(ref))
        # many pairs, several tiles of the check, one clash at the far end
        n = 700
        many = torch.stack([torch.arange(n), torch.arange(n) + n], 1).to(torch.int64)
        big = torch.zeros(2 * n + 1, 1, 16, 64, dtype=torch.bfloat16, device="cuda")
        binding.copy_blocks(big, many.cuda())
        many[n - 1, 1] = 0                                  # destination 0 is pair 0's source
        with pytest.raises(binding.PkvError) as ei:
            binding.copy_blocks(big, many.cuda())
        assert "0x20" in ei.value.message
    finally:
        binding.set_option("debug_sync", 0)
    binding.copy_blocks(d, torch.tensor([[1, 5], [2, 5]], dtype=torch.int64, device="cuda"))
    assert binding.read_device_errors() == 0              # not checked without debug sync


@pytest.mark.parametrize("kv", ["bf16", "e4m3"])
def test_prepared_decode_step_matches_the_call(kv):
    """The prepared form of pkv_decode_step (arguments marshalled once, reissued) gives
    the same cache bytes and outputs as the ordinary call, step after step."""
    w = wl.continuous_batching(seed=78, num_seqs=24, num_steps=3, median=300, cap=3000, kv_dtype=kv, poison=True)
    a, b = DeviceWorkload(w), DeviceWorkload(w)
    for k in range(len(w.steps)):
        ra = a.run_step(k, out=torch.empty_like(a.out)).clone()
        out_b = torch.empty_like(b.out)
        call = prepare_step(w, b.key_cache, b.value_cache, b.steps[k], out_b, None, True,
                            b.k_head_scales, b.v_head_scales)
        rb = call().clone()
        torch.cuda.synchronize()
        assert torch.equal(ra, rb)
        # (the caches' unused slots hold NaN: compare the bytes)
        assert torch.equal(a.key_cache.view(torch.uint8), b.key_cache.view(torch.uint8))
        assert torch.equal(a.value_cache.view(torch.uint8), b.value_cache.view(torch.uint8))
    assert binding.read_device_errors() == 0


@pytest.mark.parametrize("hq,hk,d,kv", [(32, 32, 128, "bf16"), (12, 4, 128, "bf16"), (24, 4, 64, "bf16"),
                                        (16, 16, 128, "e4m3"), (12, 2, 128, "e4m3")])
def test_tensor_kernel_groups_not_a_multiple_of_four(hq, hk, d, kv):
    """Query-head groups of 1, 3 and 6 (rows of 1 or 2 heads, the MMA tile padded) run
    on the tensor-core kernel (forced, and chosen automatically) and match the oracle."""
    w = wl.variable_length_decode(f"g{hq // hk}_{kv}_{d}", 100 + hq + hk, [1, 17, 300, 1200, 2500], hq, hk, d, 16,
                                  kv, poison=True)
    binding.set_option("decode_kernel", 2)
    try:
        forced = check_workload(w)[0]
    finally:
        binding.set_option("decode_kernel", 0)
    for x, y in zip(forced, run_device(w)[0]):
        assert torch.equal(x, y)


def test_launch_count_and_determinism(kernel):
    w = wl.llama3_8b_decode(seed=99, num_seqs=4, len_range=(600, 1500))
    dw = DeviceWorkload(w)
    n0 = binding.launch_count()
    a = dw.run_step(0, out=torch.empty_like(dw.out), joint=False).clone()
    b = dw.run_step(0, out=torch.empty_like(dw.out), joint=False).clone()   # same slot, same data
    torch.cuda.synchronize()
    # write + decode main kernel + merge of split contexts
    assert binding.launch_count() - n0 == 2 * 3
    assert torch.equal(a, b)
    # the fused append, forced, folds the write into the tensor-core kernel; the
    # CUDA-core kernel keeps the separate write
    binding.set_option("fused_append", 2)
    try:
        n0 = binding.launch_count()
        c = dw.run_step(0, out=torch.empty_like(dw.out), joint="fused").clone()
        torch.cuda.synchronize()
    finally:
        binding.set_option("fused_append", 0)
    assert binding.launch_count() - n0 == (2 if kernel == "tensor" else 3)
    assert torch.equal(a, c)


@pytest.mark.parametrize("case", ["llama3", "cb_e4m3_bs8", "cow"])
def test_decode_step_equals_write_then_decode(case, kernel):
    """The joint call and the fused append give the same bytes as the write and the
    decode issued as two calls: outputs and both caches, step after step."""
    make = {"llama3": lambda: wl.llama3_8b_decode(seed=41, num_seqs=12, len_range=(1, 1500), poison=True),
            "cb_e4m3_bs8": lambda: wl.continuous_batching(seed=42, block_size=8, kv_dtype="e4m3", num_seqs=40,
                                                          num_steps=3, median=300, cap=3000, poison=True),
            "cow": lambda: wl.shared_prefix_cow(num_groups=4, prefix_blocks=8, suffix_range=(16, 120), poison=True)}
    w = make[case]()
    runs = {}
    for joint in ("fused", "forced", True, False):
        dw = DeviceWorkload(w)
        binding.set_option("fused_append", 2 if joint == "forced" else 0)
        try:
            outs = [dw.run_step(i, out=torch.empty_like(dw.out), joint="fused" if joint == "forced" else joint).clone()
                    for i in range(len(w.steps))]
        finally:
            binding.set_option("fused_append", 0)
        torch.cuda.synchronize()
        runs[joint] = (outs, dw.key_cache.clone(), dw.value_cache.clone())
    assert binding.read_device_errors() == 0
    for joint in ("fused", "forced", True):
        for a, b in zip(runs[joint][0], runs[False][0]):
            assert torch.equal(a, b), joint
        assert torch.equal(raw(runs[joint][1]), raw(runs[False][1])), joint
        assert torch.equal(raw(runs[joint][2]), raw(runs[False][2])), joint


def test_workspace_reuse_across_shapes_and_kernels():
    """Calls with more, then fewer, then more rows share one workspace, with CUDA-core
    calls (whose partial results use it differently) in between: every call matches the
    oracle and raises no device error, so nothing is read that this call did not write
    (partials of an earlier call with similar inputs would still be close)."""
    cases = [("tensor", wl.llama3_8b_decode(seed=51, num_seqs=40, len_range=(1, 1200))),
             ("core", wl.llama3_8b_decode(seed=52, num_seqs=24, len_range=(600, 3000))),
             ("tensor", wl.llama3_8b_decode(seed=53, num_seqs=6, len_range=(1, 700))),
             ("tensor", wl.continuous_batching(seed=54, block_size=16, kv_dtype="bf16", num_seqs=160, num_steps=2,
                                               median=300, cap=3000)),
             ("core", wl.llama3_8b_decode(seed=55, num_seqs=3, len_range=(900, 2000))),
             ("tensor", wl.llama3_8b_decode(seed=56, num_seqs=64, len_range=(1, 2048)))]
    try:
        for kern, w in cases:
            binding.set_option("decode_kernel", 2 if kern == "tensor" else 1)
            binding.set_option("partition_tokens", 256 if kern == "core" else 0)
            check_workload(w)
    finally:
        binding.set_option("decode_kernel", 0)
        binding.set_option("partition_tokens", 0)


@pytest.fixture
def work_split():
    def set_(share, chunk):
        binding.set_option("dynamic_share", share)
        binding.set_option("dynamic_chunk", chunk)
    binding.set_option("decode_kernel", 2)
    yield set_
    binding.set_option("decode_kernel", 0)
    binding.set_option("dynamic_share", -1)
    binding.set_option("dynamic_chunk", 4)


@pytest.mark.parametrize("share,chunk", [(0, 4), (256, 4), (384, 4), (512, 3), (1024, 1)])
def test_tensor_kernel_work_split_settings(share, chunk, work_split):
    """How much of the work warps claim at run time changes which warp runs which
    stages, not the values: every setting matches the oracle, and launches in a row
    (the merge kernel zeroes the claim counter for the next one) give identical bits."""
    work_split(share, chunk)
    check_workload(wl.llama3_8b_decode(seed=31, num_seqs=8, len_range=(1, 900), poison=True))
    check_workload(wl.continuous_batching(block_size=8, kv_dtype="e4m3", num_seqs=24, num_steps=2,
                                          median=200, cap=2000, poison=True))
    w = wl.llama3_8b_decode(seed=32, num_seqs=64, len_range=(100, 2048))
    dw = DeviceWorkload(w)
    runs = [dw.run_step(0, out=torch.empty_like(dw.out)).clone() for _ in range(3)]
    torch.cuda.synchronize()
    assert binding.read_device_errors() == 0
    assert torch.equal(runs[0], runs[1]) and torch.equal(runs[0], runs[2])


def test_merge_of_rows_of_many_parts(work_split):
    """Rows cut into many parts (a long context in one-stage run-time units, rows of
    many sequences folded side by side in one merge block): the merge matches the
    oracle and launches in a row give identical bits."""
    work_split(1024, 1)
    check_workload(wl.long_context(num_seqs=2, context_len=20000))
    check_workload(wl.continuous_batching(block_size=16, kv_dtype="e4m3", num_seqs=40, num_steps=2,
                                          median=300, cap=3000, poison=True))
    w = wl.llama3_8b_decode(seed=33, num_seqs=64, len_range=(100, 2048))
    dw = DeviceWorkload(w)
    runs = [dw.run_step(0, out=torch.empty_like(dw.out)).clone() for _ in range(5)]
    torch.cuda.synchronize()
    assert binding.read_device_errors() == 0
    assert all(torch.equal(runs[0], r) for r in runs[1:])


def test_tensor_kernel_all_claimed_full_size(work_split):
    """Every stage claimed at run time, more units than the cap allows at one stage
    each (the kernel widens them): the full Llama-3-8B-shaped batch."""
    work_split(1024, 1)
    check_workload(wl.llama3_8b_decode())


def test_auto_selects_tensor_core_kernel_for_gqa_bf16():
    """With no override the library runs the tensor-core kernel for GQA bf16 calls:
    its output is bit-identical to the forced tensor-core run (the CUDA-core kernel
    rounds differently)."""
    w = wl.llama3_8b_decode(seed=98, num_seqs=4, len_range=(600, 1500))
    dw = DeviceWorkload(w)
    dw.run_step(0)
    outs = {}
    for k in (0, 2, 1):
        binding.set_option("decode_kernel", k)
        outs[k] = dw.run_step(0, out=torch.empty_like(dw.out)).clone()
    binding.set_option("decode_kernel", 0)
    torch.cuda.synchronize()
    assert torch.equal(outs[0], outs[2])
    assert not torch.equal(outs[0], outs[1])


def test_tensor_core_kernel_rejects_what_it_cannot_run():
    w = wl.variable_length_decode("nt", 97, [10, 20], 8, 2, 128, 4, "bf16")   # block size 4
    dw = DeviceWorkload(w)
    binding.set_option("decode_kernel", 2)
    try:
        with pytest.raises(binding.PkvError) as ei:
            dw.run_step(0)
        assert ei.value.status == 2
    finally:
        binding.set_option("decode_kernel", 0)


@pytest.mark.parametrize("bs", [8, 16, 32])
def test_prefill_over_prefix_cached_blocks(bs, pkernel):
    """Prompts sharing a system prompt's cached blocks through the prefix cache: every
    sequence of the step reads the same physical prefix blocks and prefills its own
    suffix (unused slots NaN)."""
    check_workload(wl.prefix_cached_prefill(seed=20 + bs, system_len=300, suffix_lens=(40, 1, 129, 16, 7),
                                            block_size=bs, poison=True))


@pytest.mark.parametrize("kv", ["bf16", "e4m3"])
def test_largest_batch_of_the_tensor_core_kernel(kv, kernel):
    """4096 sequences (about the most one launch of the 16-bit tensor-core kernel takes:
    its per-sequence offsets fill shared memory) of 1 to 40 tokens, unused slots NaN;
    steps as write + decode, joint, and with the in-kernel append forced (which falls
    back to two launches when its staged tokens no longer fit)."""
    w = wl.variable_length_decode(f"max_batch_{kv}", 73, torch.randint(1, 41, (4096,),
                                  generator=torch.Generator().manual_seed(73)).tolist(),
                                  32, 8, 128, 16, kv, poison=True)
    check_workload(w)
    runs = {}
    for mode in ("joint", "forced"):
        dw = DeviceWorkload(w)
        binding.set_option("fused_append", 2 if mode == "forced" else 0)
        try:
            runs[mode] = dw.run_step(0, out=torch.empty_like(dw.out), joint="fused" if mode == "forced" else True).clone()
        finally:
            binding.set_option("fused_append", 0)
        torch.cuda.synchronize()
    assert binding.read_device_errors() == 0
    assert torch.equal(runs["joint"], runs["forced"])


@pytest.mark.parametrize("kv,num_seqs", [("bf16", 4400), ("bf16", 8192), ("e4m3", 12000)])
def test_batches_past_one_launch_run_as_several(kv, num_seqs):
    """More sequences than one launch's shared memory holds offsets for: the tensor-core
    kernel (forced) runs consecutive ranges of sequences as launches of their own, in
    stream order, and matches the oracle; the automatic choice takes the same path."""
    lens = [1 + (i * 7 % 37) for i in range(num_seqs)]
    w = wl.variable_length_decode(f"past_one_launch_{kv}_{num_seqs}", 74, lens, 32, 8, 128, 16, kv, poison=True)
    binding.set_option("decode_kernel", 2)
    try:
        n0 = binding.launch_count()
        check_workload(w)
        launches = binding.launch_count() - n0
    finally:
        binding.set_option("decode_kernel", 0)
    assert launches >= 1 + 2 * 2, launches        # the write, then at least two main + merge pairs
    a = run_device(w)[0]
    for x, y in zip(a, check_workload(w)[0]):
        assert torch.equal(x, y)


@pytest.mark.parametrize("draw", range(12))
def test_random_configurations(draw):
    """Seeded random draws over the supported space: GQA group, head_dim, block size,
    cache dtype, window, per-head scales, batch size and a length mix with very short
    and block-edge contexts; two decode steps each, all against the oracle (the default
    kernel choice, so both decode kernels meet draws they take)."""
    g = torch.Generator().manual_seed(1000 + draw)
    pick = lambda xs: xs[int(torch.randint(0, len(xs), (1,), generator=g))]
    hk = pick([1, 2, 4, 8])
    group = pick([1, 3, 4, 8, 16])
    d = pick([64, 128])
    bs = pick([2, 4, 8, 16, 32])
    kv = pick(["bf16", "bf16", "e4m3", "f32"])
    if kv == "e4m3" and d == 64 and bs < 8:
        bs = 16
    q = "f32" if kv == "f32" else "bf16"
    n = int(torch.randint(1, 48, (1,), generator=g))
    lens = torch.randint(1, 900, (n,), generator=g).tolist()
    lens[0] = 1
    if n > 1:
        lens[1] = bs * int(torch.randint(1, 20, (1,), generator=g))   # ends on a block edge
    window = pick([0, 0, 0, 17, 256]) if kv != "f32" else 0
    spread = 2.0 if (kv == "e4m3" and draw % 2) else 0.0
    w = wl.variable_length_decode(f"random_{draw}", 2000 + draw, lens, hk * group, hk, d, bs, kv, q_dtype=q,
                                  num_steps=2, poison=True, window=window, head_spread=spread)
    check_workload(w)


@pytest.mark.parametrize("kv", ["bf16", "e4m3"])
def test_decode_step_replayed_from_a_cuda_graph(kv):
    """A decode step (cache write, then the decode launched as its programmatic
    dependent, then the merge) captured into a CUDA graph after the workspace was
    reserved, and replayed: the same cache bytes and outputs as the eager step."""
    w = wl.continuous_batching(seed=77, num_seqs=48, num_steps=1, median=300, cap=4000, kv_dtype=kv, poison=True)
    st = w.steps[0]
    eager = DeviceWorkload(w)
    ref = eager.run_step(0, out=torch.empty_like(eager.out)).clone()
    torch.cuda.synchronize()
    binding.reserve_workspace(binding.decode_workspace_bytes(w.num_seqs, st.query.shape[1], w.num_kv_heads,
                                                             w.head_dim, w.block_size, w.max_blocks_per_seq))
    dw = DeviceWorkload(w)
    out = torch.empty_like(dw.out)
    side = torch.cuda.Stream()
    side.wait_stream(torch.cuda.current_stream())
    with torch.cuda.stream(side):                 # warm-up outside the capture
        dw.run_step(0, out=out)
    torch.cuda.current_stream().wait_stream(side)
    torch.cuda.synchronize()
    out.zero_()
    graph = torch.cuda.CUDAGraph()
    with torch.cuda.graph(graph):
        dw.run_step(0, out=out)
    for _ in range(3):                            # the step rewrites the same slots with the same bytes
        graph.replay()
    torch.cuda.synchronize()
    assert binding.read_device_errors() == 0
    assert torch.equal(out, ref)
    assert torch.equal(raw(dw.key_cache), raw(eager.key_cache))
    assert torch.equal(raw(dw.value_cache), raw(eager.value_cache))


_THREADED_CHILD = r"""
import sys, threading, torch
from paged_kv_cache_90_gb300 import binding
from paged_kv_cache_90_gb300.decode_step import DeviceWorkload
from paged_kv_cache_90_gb300 import workloads as wl
sys.path.insert(0, sys.argv[2])
from test_gpu_parity import threaded_cases
binding.load_library()
stream = torch.cuda.Stream()
outs, errors = {}, []
def run(t):
    try:
        with torch.cuda.stream(stream):
            for key, w in threaded_cases(t):
                dw = DeviceWorkload(w)
                out = dw.run_step(0, out=torch.empty_like(dw.out))
                stream.synchronize()
                outs[key] = out.cpu()
    except Exception as e:            # reported by the parent
        errors.append(repr(e))
threads = [threading.Thread(target=run, args=(t,)) for t in range(4)]
for th in threads: th.start()
for th in threads: th.join()
assert not errors, errors
assert binding.read_device_errors() == 0
torch.save(outs, sys.argv[1])
"""


def threaded_cases(t):
    """Thread t's decodes, growing in size, so that the threads grow the (initially
    empty) workspace while the others queue work."""
    return [((t, j), wl.llama3_8b_decode(seed=600 + 10 * t + j, num_seqs=n, len_range=(1, 1200 + 400 * t)))
            for j, n in enumerate((4, 24, 64))]


def test_host_threads_share_one_workspace(tmp_path):
    """Four host threads queue decodes of growing size on one stream in a fresh process
    (so the workspace grows while other threads queue work): every output matches the
    oracle and no device check fires."""
    import subprocess
    import sys
    root = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
    path = tmp_path / "outs.pt"
    r = subprocess.run([sys.executable, "-c", _THREADED_CHILD, str(path), os.path.join(root, "tests")],
                       cwd=root, capture_output=True, text=True, timeout=600)
    assert r.returncode == 0, r.stdout[-2000:] + r.stderr[-2000:]
    outs = torch.load(path)
    for t in range(4):
        for key, w in threaded_cases(t):
            kc, vc = w.key_cache.clone(), w.value_cache.clone()
            ref = oracle.run_workload_step(w, 0, kc, vc, THREADS)
            wabs = weighted_abs_values(w, w.steps[0], kc, vc)
            assert_decode_close(outs[key].double(), ref, w, wabs)
