"""The allocation-free decode entry point (pkv_paged_attention_decode_noalloc).

It serves callers that cannot let a library allocate device memory: engines that
reserve nearly all GPU memory for their KV-cache pool and own allocator, and decode
loops that must not be synchronised by cudaMalloc/cudaFree.  It must give the same
results as pkv_paged_attention_decode, call after call, while its partial results live
in the library's fixed scratch array.  This file is collected last on purpose."""
import pytest
import torch

from paged_kv_cache_90_gb300 import binding
from paged_kv_cache_90_gb300 import build as pkv_build
from paged_kv_cache_90_gb300 import workloads as wl
from paged_kv_cache_90_gb300.decode_step import DeviceWorkload

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module", autouse=True)
def _setup():
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    pkv_build.build()
    binding.load_library()
    yield
    binding.set_option("partition_tokens", 0)


def _args(dw, st):
    w = dw.w
    return (st.query, dw.key_cache, dw.value_cache, st.block_tables, st.context_lens, w.num_kv_heads,
            w.scale, w.block_size, w.max_blocks_per_seq, w.k_scale, w.v_scale)


@pytest.mark.parametrize("kernel", ["tensor", "core"])
def test_noalloc_matches_regular_entry_point_twice_in_a_row(kernel):
    binding.set_option("partition_tokens", 256)   # split contexts, so the scratch is used
    binding.set_option("decode_kernel", 2 if kernel == "tensor" else 1)
    cases = [wl.llama3_8b_decode(seed=12, num_seqs=12, len_range=(300, 1800), poison=True),
             wl.continuous_batching(seed=15, block_size=32, kv_dtype="e4m3", num_seqs=20, num_steps=1,
                                    median=400, cap=3000, poison=True)]
    for w in cases:
        dw = DeviceWorkload(w)
        dw.run_step(0)                                # write the step's new tokens
        st = dw.steps[0]
        need = binding.decode_workspace_bytes(w.num_seqs, w.num_heads, w.num_kv_heads, w.head_dim, w.block_size,
                                              w.max_blocks_per_seq)
        assert 0 < need <= binding.noalloc_scratch_bytes()
        ref = torch.empty_like(dw.out)
        binding.paged_attention_decode(ref, *_args(dw, st))
        tol = 5e-2 if w.kv_dtype == torch.float8_e4m3fn else 2e-2
        for _ in range(2):
            got = torch.full_like(dw.out, float("nan"))
            binding.paged_attention_decode_noalloc(got, *_args(dw, st))
            torch.cuda.synchronize()
            err = (got.double() - ref.double()).abs().max().item()
            assert err <= tol, f"max abs difference {err}"
        assert binding.read_device_errors() == 0
    binding.set_option("decode_kernel", 0)


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
