"""CPU oracle for the paged decode path — TEST INFRASTRUCTURE ONLY.

Only the test suite, ``__graft_entry__.smoke()`` and the benchmark's CPU-baseline leg
may import this package.  The product path (the CUDA library and its Python binding)
never imports, links or runs it, and this package imports nothing from the product
package.  It shares no code with the CUDA path.

The arithmetic lives in ``paged_ref.c`` (plain C, IEEE binary64): decode attention
written out from its definition (gather through the block table, scores, max-shifted
softmax, weighted sum of values), the slot-mapped cache write, whole-block
copy-on-write, and the bf16 / e4m3 formats from their definitions.  This module only
compiles it with gcc and marshals arguments.
"""
from __future__ import annotations

import ctypes
import os
import subprocess
import threading

import numpy as np
import torch

_HERE = os.path.dirname(os.path.abspath(__file__))
_SRC = os.path.join(_HERE, "paged_ref.c")
_BUILD = os.path.join(_HERE, "_build")
_LIB_PATH = os.path.join(_BUILD, "liboracle_paged.so")

F32, BF16, E4M3 = 0, 1, 2
_CODES = {torch.float32: F32, torch.bfloat16: BF16, torch.float8_e4m3fn: E4M3}

_lock = threading.Lock()
_lib = None


def build(force: bool = False) -> str:
    """Compile ``paged_ref.c`` with gcc (OpenMP on, no FP contraction)."""
    os.makedirs(_BUILD, exist_ok=True)
    if (not force and os.path.exists(_LIB_PATH)
            and os.path.getmtime(_LIB_PATH) >= os.path.getmtime(_SRC)):
        return _LIB_PATH
    tmp = _LIB_PATH + f".tmp{os.getpid()}"
    cmd = ["gcc", "-O2", "-std=c99", "-fPIC", "-shared", "-fopenmp", "-ffp-contract=off",
           _SRC, "-o", tmp, "-lm"]
    subprocess.run(cmd, check=True)
    os.replace(tmp, _LIB_PATH)
    return _LIB_PATH


def _load():
    global _lib
    with _lock:
        if _lib is None:
            lib = ctypes.CDLL(build())
            i64, i32, dbl, vp = ctypes.c_int64, ctypes.c_int, ctypes.c_double, ctypes.c_void_p
            lib.orc_paged_attention_decode.restype = i32
            lib.orc_paged_attention_decode.argtypes = (
                [vp, vp, i32, vp, vp, i32, dbl, dbl, vp, vp] + [i64] * 10 + [dbl, i32])
            lib.orc_paged_attention_decode_window.restype = i32
            lib.orc_paged_attention_decode_window.argtypes = (
                [vp, vp, i32, vp, vp, i32, dbl, dbl, vp, vp] + [i64] * 10 + [dbl, i64, i32])
            lib.orc_paged_attention_decode_ex.restype = i32
            lib.orc_paged_attention_decode_ex.argtypes = (
                [vp, vp, i32, vp, vp, i32, dbl, dbl, vp, vp, vp, vp] + [i64] * 10 + [dbl, i64, i32])
            lib.orc_paged_attention_prefill.restype = i32
            lib.orc_paged_attention_prefill.argtypes = (
                [vp, vp, i32, vp, vp, i32, dbl, dbl, vp, vp, vp] + [i64] * 10 + [dbl, i32])
            lib.orc_reshape_and_cache_ex.restype = i32
            lib.orc_reshape_and_cache_ex.argtypes = (
                [vp, vp, i32, vp, vp, i32, ctypes.c_float, ctypes.c_float, vp, vp, vp, vp, vp] + [i64] * 8)
            lib.orc_reshape_and_cache.restype = i32
            lib.orc_reshape_and_cache.argtypes = (
                [vp, vp, i32, vp, vp, i32, ctypes.c_float, ctypes.c_float, vp] + [i64] * 8)
            lib.orc_copy_blocks.restype = i32
            lib.orc_copy_blocks.argtypes = [vp, i64, i64, vp, i64]
            lib.orc_e4m3_decode_array.argtypes = [vp, vp, i64]
            lib.orc_e4m3_encode_array.argtypes = [vp, vp, i64]
            lib.orc_bf16_decode_array.argtypes = [vp, vp, i64]
            lib.orc_max_threads.restype = i32
            _lib = lib
    return _lib


def _cpu(t: torch.Tensor) -> torch.Tensor:
    if t.device.type != "cpu":
        raise ValueError("the oracle takes CPU tensors")
    return t.contiguous()


def _cache_strides(cache: torch.Tensor):
    if cache.dim() != 4 or cache.stride(3) != 1:
        raise ValueError("cache must be [num_blocks, num_kv_heads, block_size, head_dim] "
                         "with a contiguous last dimension")
    return cache.stride(0), cache.stride(1), cache.stride(2)


def max_threads() -> int:
    return int(_load().orc_max_threads())


def _head_scales(x):
    """Per-KV-head scales as a contiguous float32 CPU tensor (or None)."""
    return None if x is None else torch.as_tensor(x, dtype=torch.float32).detach().cpu().contiguous()


def paged_attention_decode(query, key_cache, value_cache, block_tables, context_lens,
                           scale: float, k_scale: float = 1.0, v_scale: float = 1.0,
                           num_threads: int = 1, sliding_window: int = 0,
                           k_head_scales=None, v_head_scales=None) -> torch.Tensor:
    """Decode attention in fp64; returns a float64 tensor ``[S, Hq, D]``.  With
    ``sliding_window`` W > 0 each sequence attends to its last W positions only;
    ``k_head_scales`` / ``v_head_scales`` ([Hk]) replace the per-tensor scales."""
    lib = _load()
    q = _cpu(query)
    bt = _cpu(block_tables).to(torch.int32)
    cl = _cpu(context_lens).to(torch.int32)
    s, hq, d = q.shape
    nb, hk, bs, dk = key_cache.shape
    if dk != d or value_cache.shape != key_cache.shape or value_cache.stride() != key_cache.stride():
        raise ValueError("cache shapes disagree")
    cs = _cache_strides(key_cache)
    out = torch.zeros(s, hq, d, dtype=torch.float64)
    mb = bt.shape[1] if bt.dim() == 2 else 0
    ksh, vsh = _head_scales(k_head_scales), _head_scales(v_head_scales)
    for t in (ksh, vsh):
        if t is not None and t.numel() != hk:
            raise ValueError("head scales must have one entry per KV head")
    rc = lib.orc_paged_attention_decode_ex(
        out.data_ptr(), q.data_ptr(), _CODES[q.dtype], key_cache.data_ptr(),
        value_cache.data_ptr(), _CODES[key_cache.dtype], float(k_scale), float(v_scale),
        None if ksh is None else ksh.data_ptr(), None if vsh is None else vsh.data_ptr(),
        bt.data_ptr(), cl.data_ptr(), s, hq, hk, d, bs, nb, mb, cs[0], cs[1], cs[2],
        float(scale), int(sliding_window), int(num_threads))
    if rc != 0:
        raise ValueError(f"oracle decode failed with status {rc}")
    return out


def paged_attention_prefill(query, key_cache, value_cache, block_tables, context_lens, query_start_loc,
                            scale: float, k_scale: float = 1.0, v_scale: float = 1.0,
                            num_threads: int = 1) -> torch.Tensor:
    """Causal attention of the packed new tokens of every sequence over its cache, in
    fp64; returns ``[T, Hq, D]`` float64.  Sequence s owns query rows
    ``query_start_loc[s] .. query_start_loc[s+1]-1``, the last of its
    ``context_lens[s]`` cached positions."""
    lib = _load()
    q = _cpu(query)
    bt = _cpu(block_tables).to(torch.int32)
    cl = _cpu(context_lens).to(torch.int32)
    qsl = _cpu(query_start_loc).to(torch.int32)
    t, hq, d = q.shape
    nb, hk, bs, dk = key_cache.shape
    if dk != d or value_cache.shape != key_cache.shape or value_cache.stride() != key_cache.stride():
        raise ValueError("cache shapes disagree")
    if qsl.numel() != cl.numel() + 1 or int(qsl[-1]) != t:
        raise ValueError("query_start_loc must have num_seqs + 1 entries ending at the number of queries")
    cs = _cache_strides(key_cache)
    out = torch.zeros(t, hq, d, dtype=torch.float64)
    mb = bt.shape[1] if bt.dim() == 2 else 0
    rc = lib.orc_paged_attention_prefill(
        out.data_ptr(), q.data_ptr(), _CODES[q.dtype], key_cache.data_ptr(), value_cache.data_ptr(),
        _CODES[key_cache.dtype], float(k_scale), float(v_scale), bt.data_ptr(), cl.data_ptr(), qsl.data_ptr(),
        cl.numel(), hq, hk, d, bs, nb, mb, cs[0], cs[1], cs[2], float(scale), int(num_threads))
    if rc != 0:
        raise ValueError(f"oracle prefill failed with status {rc}")
    return out


def reshape_and_cache(key, value, key_cache, value_cache, slot_mapping,
                      k_scale: float = 1.0, v_scale: float = 1.0,
                      k_head_scales=None, v_head_scales=None, k_amax=None, v_amax=None) -> None:
    """Write new tokens' K/V into the caches in place (CPU tensors).  Per-head scales
    ([Hk]) replace the per-tensor ones; ``k_amax`` / ``v_amax`` (float64 [Hk] CPU
    tensors) are raised to the largest |x| written for each head."""
    lib = _load()
    k, v = _cpu(key), _cpu(value)
    sm = _cpu(slot_mapping).to(torch.int64)
    t, hk, d = k.shape
    nb, hk2, bs, d2 = key_cache.shape
    if hk2 != hk or d2 != d:
        raise ValueError("key / cache shapes disagree")
    cs = _cache_strides(key_cache)
    ksh, vsh = _head_scales(k_head_scales), _head_scales(v_head_scales)
    for a in (k_amax, v_amax):
        if a is not None and (a.dtype != torch.float64 or a.device.type != "cpu" or a.numel() != hk
                              or not a.is_contiguous()):
            raise ValueError("amax outputs must be contiguous float64 CPU tensors of num_kv_heads entries")
    rc = lib.orc_reshape_and_cache_ex(
        k.data_ptr(), v.data_ptr(), _CODES[k.dtype], key_cache.data_ptr(), value_cache.data_ptr(),
        _CODES[key_cache.dtype], float(k_scale), float(v_scale),
        None if ksh is None else ksh.data_ptr(), None if vsh is None else vsh.data_ptr(),
        None if k_amax is None else k_amax.data_ptr(), None if v_amax is None else v_amax.data_ptr(),
        sm.data_ptr(), t, hk, d, bs, nb, cs[0], cs[1], cs[2])
    if rc != 0:
        raise ValueError(f"oracle reshape_and_cache failed with status {rc}")


def copy_blocks(cache: torch.Tensor, pairs) -> None:
    """Whole-block copies ``cache[dst] = cache[src]`` in place (CPU tensor)."""
    lib = _load()
    if not cache.is_contiguous():
        raise ValueError("cache must be contiguous")
    p = _cpu(torch.as_tensor(pairs, dtype=torch.int64).view(-1, 2))
    nb = cache.shape[0]
    block_bytes = cache[0].numel() * cache.element_size()
    rc = lib.orc_copy_blocks(cache.data_ptr(), block_bytes, nb, p.data_ptr(), p.shape[0])
    if rc != 0:
        raise ValueError(f"oracle copy_blocks failed with status {rc}")


def e4m3_decode(codes) -> np.ndarray:
    c = np.ascontiguousarray(np.asarray(codes, dtype=np.uint8))
    out = np.empty(c.shape, dtype=np.float64)
    _load().orc_e4m3_decode_array(c.ctypes.data, out.ctypes.data, c.size)
    return out


def e4m3_encode(x) -> np.ndarray:
    a = np.ascontiguousarray(np.asarray(x, dtype=np.float32))
    out = np.empty(a.shape, dtype=np.uint8)
    _load().orc_e4m3_encode_array(a.ctypes.data, out.ctypes.data, a.size)
    return out


def bf16_decode(bits) -> np.ndarray:
    b = np.ascontiguousarray(np.asarray(bits, dtype=np.uint16))
    out = np.empty(b.shape, dtype=np.float64)
    _load().orc_bf16_decode_array(b.ctypes.data, out.ctypes.data, b.size)
    return out


def run_workload_step(w, step_index: int, key_cache, value_cache, num_threads: int = 1):
    """Apply one decode step of a workload on CPU caches, in the order the device
    runs it: copy-on-write pairs, then the new tokens' cache write, then decode.
    Mutates the caches; returns the fp64 decode output."""
    st = w.steps[step_index]
    if st.cow_pairs.numel():
        copy_blocks(key_cache, st.cow_pairs)
        copy_blocks(value_cache, st.cow_pairs)
    ksh, vsh = getattr(w, "k_head_scales", None), getattr(w, "v_head_scales", None)
    if st.slot_mapping.numel():
        reshape_and_cache(st.new_key, st.new_value, key_cache, value_cache, st.slot_mapping,
                          w.k_scale, w.v_scale, ksh, vsh)
    if getattr(st, "query_start_loc", None) is not None:   # a prefill step
        return paged_attention_prefill(st.query, key_cache, value_cache, st.block_tables, st.context_lens,
                                       st.query_start_loc, w.scale, w.k_scale, w.v_scale, num_threads)
    return paged_attention_decode(st.query, key_cache, value_cache, st.block_tables,
                                  st.context_lens, w.scale, w.k_scale, w.v_scale, num_threads,
                                  getattr(w, "sliding_window", 0), ksh, vsh)
