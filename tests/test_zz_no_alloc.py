"""The allocation-free decode entry point (pkv_paged_attention_decode_noalloc).

It serves callers that cannot let a library allocate device memory: engines that
reserve nearly all GPU memory for their KV-cache pool and own allocator, and decode
loops that must not be synchronised by cudaMalloc/cudaFree.  It must give the same
results as pkv_paged_attention_decode (bit for bit: the same kernels run on the same
inputs), call after call, while its partial results live in the library's fixed scratch
array, and it must not allocate.  This file is collected last on purpose."""
import os
import subprocess
import sys
import textwrap

import pytest
import torch

import oracle
from paged_kv_cache_90_gb300 import binding
from paged_kv_cache_90_gb300 import build as pkv_build
from paged_kv_cache_90_gb300 import workloads as wl
from paged_kv_cache_90_gb300.decode_step import DeviceWorkload
from test_gpu_parity import THREADS, assert_decode_close, weighted_abs_values

pytestmark = pytest.mark.gpu

REPO = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


@pytest.fixture(scope="module", autouse=True)
def _setup():
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    pkv_build.build()
    oracle.build()
    binding.load_library()
    yield
    binding.set_option("partition_tokens", 0)
    binding.set_option("decode_kernel", 0)


def _args(dw, st):
    w = dw.w
    return (st.query, dw.key_cache, dw.value_cache, st.block_tables, st.context_lens, w.num_kv_heads,
            w.scale, w.block_size, w.max_blocks_per_seq, w.k_scale, w.v_scale)


@pytest.mark.parametrize("kernel", ["tensor", "core"])
def test_noalloc_matches_regular_entry_point_twice_in_a_row(kernel):
    binding.set_option("partition_tokens", 256)   # split contexts, so the scratch is used
    binding.set_option("decode_kernel", 2 if kernel == "tensor" else 1)
    try:
        cases = [wl.llama3_8b_decode(seed=12, num_seqs=12, len_range=(300, 1800), poison=True),
                 wl.continuous_batching(seed=15, block_size=32, kv_dtype="e4m3", num_seqs=20, num_steps=1,
                                        median=400, cap=3000, poison=True)]
        for w in cases:
            kc0, vc0 = w.key_cache.clone(), w.value_cache.clone()
            dw = DeviceWorkload(w)
            dw.run_step(0)                                # write the step's new tokens
            st = dw.steps[0]
            need = binding.decode_workspace_bytes(w.num_seqs, w.num_heads, w.num_kv_heads, w.head_dim,
                                                  w.block_size, w.max_blocks_per_seq)
            assert 0 < need <= binding.noalloc_scratch_bytes()
            ref = torch.full_like(dw.out, float("nan"))
            binding.paged_attention_decode(ref, *_args(dw, st))
            # the oracle on the same step (its own copy of the cache, written by itself)
            want = oracle.run_workload_step(w, 0, kc0, vc0, THREADS)
            wabs = weighted_abs_values(w, w.steps[0], kc0, vc0) if w.q_dtype == torch.bfloat16 else None
            for _ in range(2):
                got = torch.full_like(dw.out, float("nan"))
                binding.paged_attention_decode_noalloc(got, *_args(dw, st))
                torch.cuda.synchronize()
                # the same kernels on the same inputs: identical bits
                assert torch.equal(got, ref), \
                    f"max abs difference {(got.double() - ref.double()).abs().max().item()}"
                assert_decode_close(got.double().cpu(), want, w, wabs)
            assert binding.read_device_errors() == 0
    finally:
        binding.set_option("decode_kernel", 0)
        binding.set_option("partition_tokens", 0)


_FRESH_PROCESS = textwrap.dedent("""
    import sys, torch
    sys.path.insert(0, {repo!r})
    from paged_kv_cache_90_gb300 import binding
    from paged_kv_cache_90_gb300 import workloads as wl
    from paged_kv_cache_90_gb300.decode_step import DeviceWorkload
    binding.load_library()
    binding.set_option("partition_tokens", 256)
    w = wl.llama3_8b_decode(seed=21, num_seqs=48, len_range=(600, 2000))
    dw = DeviceWorkload(w)
    st = dw.steps[0]
    need = binding.decode_workspace_bytes(w.num_seqs, w.num_heads, w.num_kv_heads, w.head_dim, w.block_size,
                                          w.max_blocks_per_seq)
    assert 4 << 20 <= need <= binding.noalloc_scratch_bytes(), need
    args = (st.query, dw.key_cache, dw.value_cache, st.block_tables, st.context_lens, w.num_kv_heads,
            w.scale, w.block_size, w.max_blocks_per_seq)
    outs = [torch.full_like(dw.out, float("nan")) for _ in range(3)]
    torch.cuda.synchronize()
    free0 = torch.cuda.mem_get_info()[0]
    binding.paged_attention_decode_noalloc(outs[0], *args)
    binding.paged_attention_decode_noalloc(outs[1], *args)
    torch.cuda.synchronize()
    free1 = torch.cuda.mem_get_info()[0]
    binding.paged_attention_decode(outs[2], *args)      # the regular call grows its workspace
    torch.cuda.synchronize()
    free2 = torch.cuda.mem_get_info()[0]
    assert binding.read_device_errors() == 0
    assert torch.equal(outs[0], outs[2]) and torch.equal(outs[1], outs[2])
    print("FREE", free0, free1, free2, need)
""")


def test_noalloc_first_call_in_a_fresh_process_allocates_nothing():
    """In a new process whose modules load eagerly (so the scratch array is already
    resident), the first decode calls through the no-alloc entry point leave the free
    device memory as it was, while the regular entry point's first call then takes its
    workspace (several MiB here), and all three outputs agree bit for bit."""
    env = dict(os.environ, CUDA_MODULE_LOADING="EAGER")
    r = subprocess.run([sys.executable, "-c", _FRESH_PROCESS.format(repo=REPO)], env=env, cwd=REPO,
                       capture_output=True, text=True, timeout=600)
    assert r.returncode == 0, r.stdout[-2000:] + r.stderr[-4000:]
    line = [ln for ln in r.stdout.splitlines() if ln.startswith("FREE")][-1]
    free0, free1, free2, need = (int(x) for x in line.split()[1:])
    assert free0 - free1 < 2 << 20, f"no-alloc calls took {free0 - free1} bytes of device memory"
    # the measurement sees an allocation of this size: the regular call's workspace (its
    # own need, at most the upper bound `need`) shows up
    assert free1 - free2 >= 4 << 20, f"the regular call took only {free1 - free2} bytes (bound {need})"


@pytest.mark.parametrize("kernel,s,mb", [("core", 64, 4096), ("tensor", 4096, 2)])
def test_noalloc_rejects_calls_beyond_its_scratch(kernel, s, mb):
    """A call whose split contexts would need more than the static scratch is refused
    with a message, and nothing is written."""
    binding.set_option("partition_tokens", 0)
    binding.set_option("decode_kernel", 1 if kernel == "core" else 2)
    try:
        w = wl.llama3_8b_decode(seed=13, num_seqs=4, len_range=(100, 200))
        dw = DeviceWorkload(w)
        bt = torch.zeros(s, mb, dtype=torch.int32, device="cuda")
        cl = torch.ones(s, dtype=torch.int32, device="cuda")
        q = torch.zeros(s, 32, 128, dtype=torch.bfloat16, device="cuda")
        out = torch.zeros_like(q)
        with pytest.raises(binding.PkvError) as ei:
            binding.paged_attention_decode_noalloc(out, q, dw.key_cache, dw.value_cache, bt, cl, 8, w.scale,
                                                   16, mb)
        assert ei.value.status == 1 and "scratch" in ei.value.message
        torch.cuda.synchronize()
        assert torch.all(out == 0)
    finally:
        binding.set_option("decode_kernel", 0)
