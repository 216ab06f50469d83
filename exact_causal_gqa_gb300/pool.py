"""Binding of the bounded hot-page pool (include/atlas_pool.h).

A device pool of ``hot_slots + scratch_slots`` K/V pages fed from a host tier
(CFR-Atlas README, introduction: a byte-bounded hot cache and reusable scratch
buffers for cold pages, folded into the online softmax one after another).  The
planner (policy, residency, passes) is native code in libatlas_attn.so; the copies
and the attention run in its kernels.  This module only marshals arguments and
orders the calls on the current stream.
"""
from __future__ import annotations

import ctypes
from typing import Optional, Tuple

import torch

from . import (PHASE_CHUNKS, PHASE_MERGE, AtlasError, PoolStats, _PoolConfig, _PoolRequest,
               _call, load_library, split_tokens_of, status_string, workspace_size)


class HotPagePool:
    """Hot cache + scratch slots on the device, host tier in (pinned) host memory.

    ``host_k`` / ``host_v``: [host_pages][n_kv_heads][page_tokens][head_dim] tensors of
    the attention dtype, page-locked CPU memory (``pin_memory()``) or CUDA memory.
    Host page ids index their first dimension."""

    def __init__(self, host_k: torch.Tensor, host_v: torch.Tensor, hot_slots: int,
                 scratch_slots: int, device="cuda"):
        if host_k.shape != host_v.shape or host_k.dim() != 4 or host_k.dtype != host_v.dtype:
            raise ValueError("host_k/host_v must be matching [pages][Hkv][P][D] tensors")
        if not host_k.is_contiguous() or not host_v.is_contiguous():
            raise ValueError("the host tier must be contiguous")
        if not host_k.is_cuda and not (host_k.is_pinned() and host_v.is_pinned()):
            raise ValueError("a CPU host tier must be page-locked (pin_memory())")
        self.lib = load_library()
        self.host_k, self.host_v = host_k, host_v
        self.host_pages, self.Hkv, self.P, self.D = host_k.shape
        self.hot_slots, self.scratch_slots = hot_slots, scratch_slots
        self.device = torch.device(device)
        slots = hot_slots + scratch_slots
        self.k_slots = torch.empty((slots, self.Hkv, self.P, self.D), dtype=host_k.dtype,
                                   device=self.device)
        self.v_slots = torch.empty_like(self.k_slots)
        self.page_bytes = self.Hkv * self.P * self.D * host_k.element_size()
        cfg = _PoolConfig(hot_slots, scratch_slots, self.P, self.host_pages)
        handle = ctypes.c_void_p()
        rc = self.lib.atlas_pool_create(ctypes.byref(cfg), ctypes.byref(handle))
        if rc != 0:
            raise AtlasError(rc, status_string(rc))
        self._h = handle
        self._stage: Optional[torch.Tensor] = None   # pinned staging of the pass arrays
        self._stage_free: Optional[torch.cuda.Event] = None

    def close(self):
        if getattr(self, "_h", None):
            self.lib.atlas_pool_destroy(self._h)
            self._h = None

    def __del__(self):
        self.close()

    def slot_of(self, host_page: int) -> int:
        """Hot slot holding ``host_page`` (-1 if it is not hot)."""
        return self.lib.atlas_pool_slot_of(self._h, host_page)

    def invalidate(self, host_page: int):
        """Drop ``host_page`` from the hot cache (its host-tier contents changed)."""
        self.lib.atlas_pool_invalidate(self._h, host_page)

    def plan(self, host_page_table: torch.Tensor, seq_lens: torch.Tensor, chunk_tokens: int,
             keep_recent_tokens: int = -1, admit: bool = True) -> PoolStats:
        """Run the planner alone (atlas_pool_plan) on CPU int32 tensors."""
        for name, t in (("host_page_table", host_page_table), ("seq_lens", seq_lens)):
            if t.is_cuda or t.dtype != torch.int32 or not t.is_contiguous():
                raise ValueError(f"{name} must be a contiguous int32 CPU tensor")
        req = _PoolRequest(host_page_table.shape[0], host_page_table.shape[1],
                           host_page_table.data_ptr(), seq_lens.data_ptr(), chunk_tokens,
                           keep_recent_tokens, 1 if admit else 0)
        stats = PoolStats()
        rc = self.lib.atlas_pool_plan(self._h, ctypes.byref(req), ctypes.byref(stats))
        if rc != 0:
            raise AtlasError(rc, status_string(rc))
        return stats

    def pass_arrays(self, k: int, batch: int, max_pages: int):
        """(page_table [B][MP], chunk_range [B][2], copies [n][2]) of pass k, CPU int32."""
        table = torch.empty((batch, max_pages), dtype=torch.int32)
        rng = torch.empty((batch, 2), dtype=torch.int32)
        cap = self.hot_slots + self.scratch_slots
        copies = torch.empty((cap, 2), dtype=torch.int32)
        n = ctypes.c_int32()
        rc = self.lib.atlas_pool_pass(self._h, k, table.data_ptr(), rng.data_ptr(),
                                      copies.data_ptr(), cap, ctypes.byref(n))
        if rc != 0:
            raise AtlasError(rc, status_string(rc))
        return table, rng, copies[:n.value]

    def fill(self, copies: torch.Tensor, status: Optional[torch.Tensor] = None):
        """Copy the listed (host page, slot) pairs in (atlas_pool_fill); ``copies``
        is an int32 CUDA tensor [n][2]."""
        n = copies.shape[0]
        if n == 0:
            return
        stream = torch.cuda.current_stream(self.device).cuda_stream
        rc = self.lib.atlas_pool_fill(self.host_k.data_ptr(), self.host_v.data_ptr(),
                                      self.k_slots.data_ptr(), self.v_slots.data_ptr(),
                                      copies.data_ptr(), n, self.page_bytes, self.host_pages,
                                      self.k_slots.shape[0],
                                      None if status is None else status.data_ptr(), stream)
        if rc != 0:
            raise AtlasError(rc, status_string(rc))

    def decode(self, q: torch.Tensor, host_page_table: torch.Tensor, seq_lens: torch.Tensor,
               n_q_heads: int, scale: float, *, keep_recent_tokens: int = -1,
               admit: bool = True, out: Optional[torch.Tensor] = None, out_dtype=None,
               lse: Optional[torch.Tensor] = None, status: Optional[torch.Tensor] = None,
               workspace: Optional[torch.Tensor] = None,
               split_tokens: int = 0) -> Tuple[torch.Tensor, PoolStats]:
        """One decode step over the pool: plan, then per pass copy in and compute its
        chunks, then merge.  ``q`` [B][Hq][1][D] on the device; ``host_page_table``
        [B][MP] and ``seq_lens`` [B] int32 on the CPU.  The result equals
        atlas_attn_decode over a pool holding every page, bit for bit."""
        B, MP = host_page_table.shape
        slots = self.k_slots.shape[0]
        dtype = self.k_slots.dtype
        out_dtype = out_dtype or (out.dtype if out is not None else q.dtype)
        chunk = split_tokens_of("decode", q.shape, n_q_heads, self.Hkv, self.D, self.P, MP,
                                slots, dtype, out_dtype, split_tokens=split_tokens,
                                phase=PHASE_CHUNKS)
        stats = self.plan(host_page_table, seq_lens, chunk, keep_recent_tokens, admit)
        npass = stats.passes
        cap = self.hot_slots + self.scratch_slots
        per = B * MP + 2 * B + 2 * cap
        need = B + npass * per
        if self._stage_free is not None:
            self._stage_free.synchronize()  # the previous call's copy has read the stage
        if self._stage is None or self._stage.numel() < need:
            self._stage = torch.empty(need, dtype=torch.int32, pin_memory=True)
        st = self._stage
        st[:B].copy_(seq_lens)
        counts = []
        ncop = ctypes.c_int32()
        for k in range(npass):
            base = B + k * per
            rc = self.lib.atlas_pool_pass(self._h, k, st[base:].data_ptr(),
                                          st[base + B * MP:].data_ptr(),
                                          st[base + B * MP + 2 * B:].data_ptr(), cap,
                                          ctypes.byref(ncop))
            if rc != 0:
                raise AtlasError(rc, status_string(rc))
            counts.append(ncop.value)
        dev = st[:need].to(self.device, non_blocking=True)
        if self._stage_free is None:
            self._stage_free = torch.cuda.Event()
        self._stage_free.record(torch.cuda.current_stream(self.device))
        seq_dev = dev[:B]
        if workspace is None:
            n = workspace_size("decode", q.shape, n_q_heads, self.Hkv, self.D, self.P, MP,
                               slots, dtype, out_dtype, split_tokens=split_tokens,
                               phase=PHASE_CHUNKS)
            workspace = torch.empty(max(n, 16), dtype=torch.uint8, device=self.device)
        for k in range(npass):
            base = B + k * per
            table = dev[base:base + B * MP].view(B, MP)
            rng = dev[base + B * MP:base + B * MP + 2 * B].view(B, 2)
            copies = dev[base + B * MP + 2 * B:base + B * MP + 2 * B + 2 * counts[k]].view(-1, 2)
            self.fill(copies, status)
            _call("decode", q, self.k_slots, self.v_slots, table, seq_dev, n_q_heads, self.Hkv,
                  self.D, self.P, scale, out_dtype=out_dtype, status=status,
                  workspace=workspace, split_tokens=split_tokens, chunk_range=rng,
                  phase=PHASE_CHUNKS)
        table0 = dev[B:B + B * MP].view(B, MP)
        out = _call("decode", q, self.k_slots, self.v_slots, table0, seq_dev, n_q_heads,
                    self.Hkv, self.D, self.P, scale, out=out, out_dtype=out_dtype, lse=lse,
                    status=status, workspace=workspace, split_tokens=split_tokens,
                    phase=PHASE_MERGE)
        return out, stats
