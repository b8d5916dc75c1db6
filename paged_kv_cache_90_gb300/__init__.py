"""GB300-native PagedAttention decode: a paged K/V cache and its hot path
(slot-mapped cache write, copy-on-write block copy, paged decode attention) as
hand-written CUDA kernels behind a C ABI (include/pkv.h, libpkv.so).

``binding`` holds the ctypes entry points; ``block_manager`` the host-side block
pool and tables; ``workloads`` the seeded synthetic inputs.
"""
from .binding import (PkvError, copy_blocks, decode_append, decode_step, decode_workspace_bytes,  # noqa: F401
                      get_option, launch_count, load_library, paged_attention_decode,
                      paged_attention_decode_noalloc, paged_attention_prefill, read_device_errors,
                      reserve_workspace, reshape_and_cache, set_option)
