"""ctypes binding of libpkv (include/pkv.h).

Argument marshalling only: each function turns torch tensors into pkv_tensor
descriptors (device pointer, dtype, shape, strides, fp8 scale), passes the current
CUDA stream, and raises :class:`PkvError` on a non-OK status.  Every step of the work
runs in the library's CUDA kernels; if the library is not built this module raises
instead of falling back to anything else.
"""
from __future__ import annotations

import ctypes
import os
import threading
from typing import Optional

import torch

_HERE = os.path.dirname(os.path.abspath(__file__))
LIB_PATH = os.path.join(_HERE, "_build", "libpkv.so")

PKV_OK = 0
STATUS_NAMES = {0: "PKV_OK", 1: "PKV_ERR_INVALID_ARG", 2: "PKV_ERR_UNSUPPORTED", 3: "PKV_ERR_CUDA",
                4: "PKV_ERR_DEVICE_CHECK"}
DEVERR = {"table_entry": 0x1, "slot": 0x2, "copy_pair": 0x4, "context_len": 0x8, "timeout": 0x10,
          "copy_overlap": 0x20}
OPTIONS = {"partition_tokens": 0, "debug_sync": 1, "dry_run": 2, "decode_kernel": 3,
           "dynamic_share": 4, "dynamic_chunk": 5, "fused_append": 6,
           "prefill_kernel": 7}
_DTYPES = {torch.float32: 0, torch.bfloat16: 1, torch.float8_e4m3fn: 2, torch.int32: 3, torch.int64: 4}


class PkvError(RuntimeError):
    def __init__(self, status: int, message: str):
        super().__init__(f"{STATUS_NAMES.get(status, status)}: {message}")
        self.status = status
        self.message = message


class PkvTensor(ctypes.Structure):
    _fields_ = [("data", ctypes.c_void_p), ("dtype", ctypes.c_int32), ("ndim", ctypes.c_int32),
                ("shape", ctypes.c_int64 * 4), ("stride", ctypes.c_int64 * 4), ("scale", ctypes.c_float),
                ("head_scales", ctypes.c_void_p)]


_lock = threading.Lock()
_lib = None


def load_library(path: Optional[str] = None) -> ctypes.CDLL:
    """Load libpkv.so (built in-tree by paged_kv_cache_90_gb300.build)."""
    global _lib
    with _lock:
        if _lib is not None:
            return _lib
        p = path or LIB_PATH
        if not os.path.exists(p):
            raise RuntimeError(f"{p} is missing: build it with `python -m paged_kv_cache_90_gb300.build` "
                               "(or __graft_entry__.build()); there is no fallback path")
        lib = ctypes.CDLL(p)
        d = ctypes.POINTER(PkvTensor)
        i32, i64, f32, vp = ctypes.c_int32, ctypes.c_int64, ctypes.c_float, ctypes.c_void_p
        lib.pkv_paged_attention_decode.argtypes = [d, d, d, d, d, d, i32, f32, i32, i32, vp]
        lib.pkv_reshape_and_cache.argtypes = [d, d, d, d, d, vp]
        lib.pkv_copy_blocks.argtypes = [d, d, vp]
        lib.pkv_paged_attention_decode_noalloc.argtypes = [d, d, d, d, d, d, i32, f32, i32, i32, vp]
        lib.pkv_decode_step.argtypes = [d, d, d, d, d, d, d, d, d, i32, f32, i32, i32, i32, vp]
        lib.pkv_reshape_and_cache_amax.argtypes = [d, d, d, d, d, vp, vp, vp]
        lib.pkv_paged_attention_prefill.argtypes = [d, d, d, d, d, d, d, i32, f32, i32, i32, vp]
        lib.pkv_decode_append.argtypes = [d, d, d, d, d, d, d, d, d, i32, f32, i32, i32, i32, vp]
        lib.pkv_paged_attention_decode_window.argtypes = [d, d, d, d, d, d, i32, f32, i32, i32, i32, vp]
        lib.pkv_noalloc_scratch_bytes.restype = i64
        lib.pkv_noalloc_scratch_bytes.argtypes = []
        for fn in ("pkv_paged_attention_decode", "pkv_paged_attention_decode_noalloc",
                   "pkv_reshape_and_cache", "pkv_decode_step", "pkv_copy_blocks",
                   "pkv_paged_attention_decode_window", "pkv_reshape_and_cache_amax",
                   "pkv_paged_attention_prefill", "pkv_decode_append",
                   "pkv_set_option", "pkv_reserve_workspace", "pkv_read_device_errors"):
            getattr(lib, fn).restype = ctypes.c_int
        lib.pkv_last_error.restype = ctypes.c_char_p
        lib.pkv_last_error.argtypes = []
        lib.pkv_abi_version.restype = i32
        lib.pkv_set_option.argtypes = [i32, i64]
        lib.pkv_get_option.restype = i64
        lib.pkv_get_option.argtypes = [i32]
        lib.pkv_reserve_workspace.argtypes = [i64]
        lib.pkv_decode_workspace_bytes.restype = i64
        lib.pkv_decode_workspace_bytes.argtypes = [i32, i32, i32, i32, i32, i32]
        lib.pkv_read_device_errors.argtypes = [ctypes.POINTER(ctypes.c_uint32)]
        lib.pkv_launch_count.restype = ctypes.c_uint64
        lib.pkv_launch_count.argtypes = []
        _lib = lib
        return lib


def _check(status: int) -> None:
    if status != PKV_OK:
        msg = load_library().pkv_last_error()
        raise PkvError(status, msg.decode() if msg else "")


def describe(t: torch.Tensor, scale: float = 1.0, head_scales: Optional[torch.Tensor] = None) -> PkvTensor:
    """pkv_tensor descriptor of a tensor (pointer, dtype code, shape, strides); an 8-bit
    cache may carry one scale per KV head (a float32 tensor on the cache's device)."""
    if t.dim() > 4 or t.dim() < 1:
        raise ValueError("descriptors cover 1 to 4 dimensions")
    if t.dtype not in _DTYPES:
        raise TypeError(f"dtype {t.dtype} has no pkv code")
    d = PkvTensor()
    d.data = t.data_ptr() if t.numel() else None
    d.dtype = _DTYPES[t.dtype]
    d.ndim = t.dim()
    for i in range(4):
        d.shape[i] = t.shape[i] if i < t.dim() else 1
        d.stride[i] = t.stride(i) if i < t.dim() else 1
    d.scale = float(scale)
    if head_scales is not None:
        if head_scales.dtype != torch.float32 or not head_scales.is_contiguous() or head_scales.device != t.device:
            raise ValueError("head scales must be a contiguous float32 tensor on the cache's device")
        d.head_scales = head_scales.data_ptr()
    return d


# Descriptors the call wrappers pass, by everything a descriptor holds (address, dtype,
# shape, strides, scale, per-head scales): a serving loop passes the same tensors every
# step, and building a descriptor costs several microseconds of Python.  The cached
# objects never leave this module, so nothing mutates them.
_DESC_CACHE: dict = {}
_DESC_CACHE_MAX = 4096


def _ref(t: torch.Tensor, scale: float = 1.0, head_scales: Optional[torch.Tensor] = None):
    hs = None if head_scales is None else (head_scales.data_ptr(), head_scales.dtype, head_scales.device,
                                             head_scales.stride())
    key = (t.data_ptr(), t.dtype, t.device, t.shape, t.stride(), float(scale), hs)
    r = _DESC_CACHE.get(key)
    if r is None:
        if len(_DESC_CACHE) >= _DESC_CACHE_MAX:
            _DESC_CACHE.clear()
        r = _DESC_CACHE[key] = ctypes.byref(describe(t, scale, head_scales))
    return r


def _stream(stream) -> ctypes.c_void_p:
    if stream is None:
        if not torch.cuda.is_available():
            return ctypes.c_void_p(0)
        stream = torch.cuda.current_stream()
    if isinstance(stream, torch.cuda.Stream):
        return ctypes.c_void_p(stream.cuda_stream)
    return ctypes.c_void_p(int(stream))


def paged_attention_decode(out, query, key_cache, value_cache, block_tables, context_lens,
                           num_kv_heads: int, scale: float, block_size: int,
                           max_blocks_per_seq: int, k_scale: float = 1.0, v_scale: float = 1.0,
                           stream=None, sliding_window: int = 0, k_head_scales=None,
                           v_head_scales=None) -> torch.Tensor:
    """Single-token decode attention over the paged cache into ``out`` (returned).
    ``sliding_window`` W > 0: each sequence attends to its last W positions only
    (pkv_paged_attention_decode_window).  ``k_head_scales`` / ``v_head_scales``: one
    scale per KV head of an 8-bit cache (device float32), instead of k_scale / v_scale."""
    lib = load_library()
    descs = [_ref(out), _ref(query), _ref(key_cache, k_scale, k_head_scales),
             _ref(value_cache, v_scale, v_head_scales), _ref(block_tables), _ref(context_lens)]
    if sliding_window:
        _check(lib.pkv_paged_attention_decode_window(*descs, int(num_kv_heads), float(scale), int(block_size),
                                                     int(max_blocks_per_seq), int(sliding_window),
                                                     _stream(stream)))
    else:
        _check(lib.pkv_paged_attention_decode(*descs, int(num_kv_heads), float(scale), int(block_size),
                                              int(max_blocks_per_seq), _stream(stream)))
    return out


def decode_step(out, query, key, value, slot_mapping, key_cache, value_cache, block_tables, context_lens,
                num_kv_heads: int, scale: float, block_size: int, max_blocks_per_seq: int,
                k_scale: float = 1.0, v_scale: float = 1.0, stream=None,
                sliding_window: int = 0, k_head_scales=None, v_head_scales=None) -> torch.Tensor:
    """Append the step's new tokens (``key``/``value`` at ``slot_mapping``) to the cache
    and decode into ``out`` (returned): the results of reshape_and_cache followed by
    paged_attention_decode, with the decode's preparation overlapping the write."""
    lib = load_library()
    descs = [_ref(out), _ref(query), _ref(key), _ref(value), _ref(slot_mapping),
             _ref(key_cache, k_scale, k_head_scales), _ref(value_cache, v_scale, v_head_scales),
             _ref(block_tables), _ref(context_lens)]
    _check(lib.pkv_decode_step(*descs, int(num_kv_heads), float(scale),
                               int(block_size), int(max_blocks_per_seq), int(sliding_window), _stream(stream)))
    return out


def prepare_decode_step(out, query, key, value, slot_mapping, key_cache, value_cache, block_tables,
                        context_lens, num_kv_heads: int, scale: float, block_size: int, max_blocks_per_seq: int,
                        k_scale: float = 1.0, v_scale: float = 1.0, stream=None, sliding_window: int = 0,
                        k_head_scales=None, v_head_scales=None):
    """decode_step's arguments marshalled once: the returned callable issues that same
    call (same tensors, same stream, resolved now) each time it is called, with nothing
    rebuilt, for serving loops that reuse their buffers every step.  The tensors must
    stay alive, on the same storage, shapes and strides, while the callable is used (it
    holds references to them).  Each call returns ``out``."""
    lib = load_library()
    keep = (out, query, key, value, slot_mapping, key_cache, value_cache, block_tables, context_lens,
            k_head_scales, v_head_scales)
    descs = [describe(out), describe(query), describe(key), describe(value), describe(slot_mapping),
             describe(key_cache, k_scale, k_head_scales), describe(value_cache, v_scale, v_head_scales),
             describe(block_tables), describe(context_lens)]
    args = tuple(ctypes.byref(d) for d in descs) + (
        ctypes.c_int32(int(num_kv_heads)), ctypes.c_float(float(scale)), ctypes.c_int32(int(block_size)),
        ctypes.c_int32(int(max_blocks_per_seq)), ctypes.c_int32(int(sliding_window)), _stream(stream))
    fn = lib.pkv_decode_step

    def call() -> torch.Tensor:
        _check(fn(*args))
        return out

    call.tensors, call.descriptors = keep, descs  # kept alive with the callable
    return call


def decode_append(out, query, key, value, slot_mapping, key_cache, value_cache, block_tables, context_lens,
                  num_kv_heads: int, scale: float, block_size: int, max_blocks_per_seq: int,
                  k_scale: float = 1.0, v_scale: float = 1.0, stream=None, sliding_window: int = 0,
                  k_head_scales=None, v_head_scales=None) -> torch.Tensor:
    """decode_step for one new token per sequence (token s of ``key`` / ``value`` is
    sequence s's newest, its slot the position context_lens[s] - 1); with the
    ``fused_append`` option at 2 the write runs inside the decode kernel.  Returns
    ``out``."""
    lib = load_library()
    descs = [_ref(out), _ref(query), _ref(key), _ref(value), _ref(slot_mapping),
             _ref(key_cache, k_scale, k_head_scales), _ref(value_cache, v_scale, v_head_scales),
             _ref(block_tables), _ref(context_lens)]
    _check(lib.pkv_decode_append(*descs, int(num_kv_heads), float(scale),
                                 int(block_size), int(max_blocks_per_seq), int(sliding_window), _stream(stream)))
    return out


def paged_attention_prefill(out, query, key_cache, value_cache, block_tables, context_lens, query_start_loc,
                            num_kv_heads: int, scale: float, block_size: int, max_blocks_per_seq: int,
                            stream=None) -> torch.Tensor:
    """Causal attention of the packed new tokens of every sequence (rows
    query_start_loc[s] .. query_start_loc[s+1]-1, the last of its context_lens[s]
    cached positions) over the paged cache, into ``out`` (returned)."""
    lib = load_library()
    descs = [_ref(out), _ref(query), _ref(key_cache), _ref(value_cache), _ref(block_tables),
             _ref(context_lens), _ref(query_start_loc)]
    _check(lib.pkv_paged_attention_prefill(*descs, int(num_kv_heads), float(scale),
                                           int(block_size), int(max_blocks_per_seq), _stream(stream)))
    return out


def paged_attention_decode_noalloc(out, query, key_cache, value_cache, block_tables, context_lens,
                                   num_kv_heads: int, scale: float, block_size: int,
                                   max_blocks_per_seq: int, k_scale: float = 1.0,
                                   v_scale: float = 1.0, stream=None) -> torch.Tensor:
    """Decode attention that allocates no device memory: partial results of split
    contexts go to the library's fixed 16 MiB scratch array instead of a workspace
    grown with cudaMalloc (for callers that own all device memory, or must not let
    an allocation synchronise the device).  Calls on one device share that scratch,
    so calls on unordered streams must not overlap."""
    lib = load_library()
    descs = [_ref(out), _ref(query), _ref(key_cache, k_scale),
             _ref(value_cache, v_scale), _ref(block_tables), _ref(context_lens)]
    _check(lib.pkv_paged_attention_decode_noalloc(*descs,
                                                  int(num_kv_heads), float(scale), int(block_size),
                                                  int(max_blocks_per_seq), _stream(stream)))
    return out


def noalloc_scratch_bytes() -> int:
    return int(load_library().pkv_noalloc_scratch_bytes())


def reshape_and_cache(key, value, key_cache, value_cache, slot_mapping, k_scale: float = 1.0,
                      v_scale: float = 1.0, stream=None, k_head_scales=None, v_head_scales=None,
                      k_amax=None, v_amax=None) -> None:
    """Write the new tokens' K/V into their cache slots (in place).  ``k_amax`` /
    ``v_amax`` (device float32 [Hk], starting >= 0) are raised to the largest |x|
    written per KV head (pkv_reshape_and_cache_amax)."""
    lib = load_library()
    descs = [_ref(key), _ref(value), _ref(key_cache, k_scale, k_head_scales),
             _ref(value_cache, v_scale, v_head_scales), _ref(slot_mapping)]
    if k_amax is None and v_amax is None:
        _check(lib.pkv_reshape_and_cache(*descs, _stream(stream)))
        return
    for a in (k_amax, v_amax):
        if a is not None and (a.dtype != torch.float32 or not a.is_contiguous() or a.device != key_cache.device):
            raise ValueError("amax arrays must be contiguous float32 tensors on the cache's device")
    _check(lib.pkv_reshape_and_cache_amax(*descs, None if k_amax is None else ctypes.c_void_p(k_amax.data_ptr()),
                                          None if v_amax is None else ctypes.c_void_p(v_amax.data_ptr()),
                                          _stream(stream)))


def copy_blocks(cache, src_dst_pairs, stream=None) -> None:
    """cache[dst] = cache[src] for every (src, dst) row of ``src_dst_pairs``."""
    lib = load_library()
    pairs = src_dst_pairs
    if pairs.numel() == 0:
        pairs = pairs.reshape(0, 2)
    descs = [_ref(cache), _ref(pairs)]
    _check(lib.pkv_copy_blocks(*descs, _stream(stream)))


def set_option(name: str, value: int) -> None:
    _check(load_library().pkv_set_option(OPTIONS[name], int(value)))


def get_option(name: str) -> int:
    return int(load_library().pkv_get_option(OPTIONS[name]))


def reserve_workspace(nbytes: int) -> None:
    _check(load_library().pkv_reserve_workspace(int(nbytes)))


def decode_workspace_bytes(num_seqs, num_heads, num_kv_heads, head_dim, block_size, max_blocks_per_seq) -> int:
    return int(load_library().pkv_decode_workspace_bytes(num_seqs, num_heads, num_kv_heads, head_dim, block_size,
                                                         max_blocks_per_seq))


def read_device_errors() -> int:
    """Synchronise the current device, return and clear its error word."""
    flags = ctypes.c_uint32(0)
    _check(load_library().pkv_read_device_errors(ctypes.byref(flags)))
    return int(flags.value)


def launch_count() -> int:
    return int(load_library().pkv_launch_count())


def abi_version() -> int:
    return int(load_library().pkv_abi_version())
