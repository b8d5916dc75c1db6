"""One decode step of a serving engine, on the device, through the C ABI.

A step is the whole hot path for one batch: copy-on-write block copies (if any
sequence writes into a shared block), the new tokens' cache write, then decode
attention over every sequence's paged context (vasteelab.pages.dev
"PagedAttentionとは？", section "PagedAttentionはAttention kernelとmemory managerの
組み合わせである": the scheduler reserves blocks, the runner hands the mapping to the
kernels).  This module only moves tensors and calls :mod:`binding`; every step runs in
the library's kernels.
"""
from __future__ import annotations

from dataclasses import dataclass
from typing import List, Optional

import torch

from . import binding
from .workloads import DecodeStep, Workload


@dataclass
class DeviceStep:
    query: torch.Tensor
    new_key: torch.Tensor
    new_value: torch.Tensor
    slot_mapping: torch.Tensor
    block_tables: torch.Tensor
    context_lens: torch.Tensor
    cow_pairs: torch.Tensor
    query_start_loc: Optional[torch.Tensor] = None   # prefill steps only

    @staticmethod
    def from_host(st: DecodeStep, device, pin: bool = False) -> "DeviceStep":
        def mv(t):
            return None if t is None else t.to(device, non_blocking=pin)
        return DeviceStep(*(mv(getattr(st, f, None)) for f in DeviceStep.__dataclass_fields__))


class DeviceWorkload:
    """A workload's caches and step inputs resident on one GPU."""

    def __init__(self, w: Workload, device: str = "cuda"):
        self.w = w
        self.device = torch.device(device)
        self.key_cache = w.key_cache.to(self.device)
        self.value_cache = w.value_cache.to(self.device)
        # an 8-bit cache with one scale per KV head keeps the scales on the device
        self.k_head_scales = None if w.k_head_scales is None else w.k_head_scales.to(self.device)
        self.v_head_scales = None if w.v_head_scales is None else w.v_head_scales.to(self.device)
        self.steps: List[DeviceStep] = [DeviceStep.from_host(st, self.device) for st in w.steps]
        s, hq, d = w.steps[0].query.shape   # (packed query rows for a prefill)
        self.out = torch.empty(s, hq, d, dtype=w.q_dtype, device=self.device)

    def run_step(self, i: int, out: Optional[torch.Tensor] = None, stream=None,
                 step: Optional[DeviceStep] = None, joint=True) -> torch.Tensor:
        """Run step ``i`` (or the given device-resident inputs) on the current
        stream; returns the decode output tensor.  ``joint``: "fused" issues the step as
        one decode_append call (one new token per sequence; the write inside the decode
        kernel when the fused_append option is 2), True (the default) as one
        decode_step call, False as a write and a decode call."""
        st = step if step is not None else self.steps[i]
        out = self.out if out is None else out
        run_decode_step(self.w, self.key_cache, self.value_cache, st, out, stream, joint,
                        self.k_head_scales, self.v_head_scales)
        return out


def prepare_step(w: Workload, key_cache, value_cache, st: DeviceStep, out, stream=None, joint=True,
                 k_head_scales=None, v_head_scales=None):
    """A callable that runs the step as run_decode_step does.  A joint decode step with no
    copy-on-write pairs is marshalled once (binding.prepare_decode_step); other steps
    call run_decode_step each time."""
    if joint is True and st.query_start_loc is None and not st.cow_pairs.numel():
        return binding.prepare_decode_step(out, st.query, st.new_key, st.new_value, st.slot_mapping, key_cache,
                                           value_cache, st.block_tables, st.context_lens, w.num_kv_heads, w.scale,
                                           w.block_size, w.max_blocks_per_seq, w.k_scale, w.v_scale, stream,
                                           w.sliding_window, k_head_scales, v_head_scales)
    return lambda: run_decode_step(w, key_cache, value_cache, st, out, stream, joint, k_head_scales, v_head_scales)


def run_decode_step(w: Workload, key_cache, value_cache, st: DeviceStep, out, stream=None,
                    joint=True, k_head_scales=None, v_head_scales=None) -> None:
    if st.cow_pairs.numel():
        binding.copy_blocks(key_cache, st.cow_pairs, stream)
        binding.copy_blocks(value_cache, st.cow_pairs, stream)
    if st.query_start_loc is not None:   # prefill: write every new token, then attend causally
        if st.slot_mapping.numel():
            binding.reshape_and_cache(st.new_key, st.new_value, key_cache, value_cache, st.slot_mapping,
                                      w.k_scale, w.v_scale, stream, k_head_scales, v_head_scales)
        binding.paged_attention_prefill(out, st.query, key_cache, value_cache, st.block_tables, st.context_lens,
                                        st.query_start_loc, w.num_kv_heads, w.scale, w.block_size,
                                        w.max_blocks_per_seq, stream)
        return
    if joint == "fused" and st.slot_mapping.numel() == st.query.shape[0]:
        binding.decode_append(out, st.query, st.new_key, st.new_value, st.slot_mapping, key_cache, value_cache,
                              st.block_tables, st.context_lens, w.num_kv_heads, w.scale, w.block_size,
                              w.max_blocks_per_seq, w.k_scale, w.v_scale, stream, w.sliding_window,
                              k_head_scales, v_head_scales)
        return
    if joint:
        binding.decode_step(out, st.query, st.new_key, st.new_value, st.slot_mapping, key_cache, value_cache,
                            st.block_tables, st.context_lens, w.num_kv_heads, w.scale, w.block_size,
                            w.max_blocks_per_seq, w.k_scale, w.v_scale, stream, w.sliding_window,
                            k_head_scales, v_head_scales)
        return
    if st.slot_mapping.numel():
        binding.reshape_and_cache(st.new_key, st.new_value, key_cache, value_cache, st.slot_mapping,
                                  w.k_scale, w.v_scale, stream, k_head_scales, v_head_scales)
    binding.paged_attention_decode(out, st.query, key_cache, value_cache, st.block_tables,
                                   st.context_lens, w.num_kv_heads, w.scale, w.block_size,
                                   w.max_blocks_per_seq, w.k_scale, w.v_scale, stream, w.sliding_window,
                                   k_head_scales, v_head_scales)
