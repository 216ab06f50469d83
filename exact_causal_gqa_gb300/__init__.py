"""Exact causal grouped-query attention over paged K/V on GB300 (sm_103a).

Python binding of ``libatlas_attn.so`` (C ABI in ``include/atlas_attn.h``).
This module only marshals arguments: it checks tensor shapes and dtypes,
allocates outputs and workspace with torch, and passes raw device pointers and
the current torch stream to the library.  Every step of the computation runs in
the library's CUDA kernels; there is no CPU or torch fallback, and the import
fails loudly when the library has not been built.

Functions (same names as the C entry points):
  decode(...)   one query row per sequence            -> atlas_attn_decode
  suffix(...)   the last q_len positions as queries   -> atlas_attn_suffix
  prefill(...)  causal self-attention of a prompt     -> atlas_attn_prefill
  kv_append(...)  new tokens' K/V into their pages    -> atlas_kv_append
  workspace_size(kind, ...)                            -> atlas_attn_workspace_size
  run_host(kind, ...)  host tensors in, host tensor out (copies on the stream)
"""
from __future__ import annotations

import ctypes
import os
from typing import Optional

import torch

from . import _build

__all__ = ["AtlasError", "decode", "suffix", "prefill", "kv_append", "workspace_size", "run_host",
           "library_path", "DEV_BAD_PAGE", "DEV_BAD_SEQLEN", "DEV_TIMEOUT",
           "DEBUG_WITHHOLD_STAGE", "KIND_DECODE", "KIND_SUFFIX", "KIND_PREFILL"]

KIND_DECODE, KIND_SUFFIX, KIND_PREFILL = 0, 1, 2
_KINDS = {"decode": KIND_DECODE, "suffix": KIND_SUFFIX, "prefill": KIND_PREFILL}
DEV_BAD_PAGE, DEV_BAD_SEQLEN, DEV_TIMEOUT = 1, 2, 4
DEBUG_WITHHOLD_STAGE = 1
DEBUG_TC_DIRECT = 2
_F32, _BF16 = 0, 1
_DTYPES = {torch.float32: _F32, torch.bfloat16: _BF16}
STATUS_NAMES = {0: "ATLAS_OK", 1: "ATLAS_ERR_INVALID_ARG", 2: "ATLAS_ERR_UNSUPPORTED",
                3: "ATLAS_ERR_WORKSPACE", 4: "ATLAS_ERR_CUDA", 5: "ATLAS_ERR_DEVICE"}


class AtlasError(RuntimeError):
    """A non-OK status from the library."""

    def __init__(self, status: int, message: str):
        super().__init__(f"{STATUS_NAMES.get(status, status)}: {message}")
        self.status = status


class _Launch(ctypes.Structure):
    _fields_ = [("batch", ctypes.c_int32), ("max_pages_per_seq", ctypes.c_int32),
                ("num_pages", ctypes.c_int32), ("q_len", ctypes.c_int32),
                ("q_dtype", ctypes.c_int), ("kv_dtype", ctypes.c_int),
                ("out_dtype", ctypes.c_int), ("out", ctypes.c_void_p),
                ("lse", ctypes.c_void_p), ("workspace", ctypes.c_void_p),
                ("workspace_bytes", ctypes.c_size_t), ("status_word", ctypes.c_void_p),
                ("stream", ctypes.c_void_p), ("split_tokens", ctypes.c_int32),
                ("debug_flags", ctypes.c_uint32), ("events", ctypes.c_void_p),
                ("window", ctypes.c_int32), ("softcap", ctypes.c_float),
                ("sinks", ctypes.c_void_p), ("q_lens", ctypes.c_void_p),
                ("chunk_range", ctypes.c_void_p), ("phase", ctypes.c_int32),
                ("sm_count", ctypes.c_int32)]

PHASE_ALL, PHASE_CHUNKS, PHASE_MERGE = 0, 1, 2


class _PoolConfig(ctypes.Structure):
    _fields_ = [("hot_slots", ctypes.c_int32), ("scratch_slots", ctypes.c_int32),
                ("page_tokens", ctypes.c_int32), ("host_pages", ctypes.c_int32)]


class _PoolRequest(ctypes.Structure):
    _fields_ = [("batch", ctypes.c_int32), ("max_pages_per_seq", ctypes.c_int32),
                ("host_page_table", ctypes.c_void_p), ("seq_lens", ctypes.c_void_p),
                ("chunk_tokens", ctypes.c_int32), ("keep_recent_tokens", ctypes.c_int32),
                ("admit", ctypes.c_int32)]


class PoolStats(ctypes.Structure):
    """What one plan of a HotPagePool did (atlas_pool_stats)."""
    _fields_ = [("passes", ctypes.c_int32), ("pages", ctypes.c_int64), ("hits", ctypes.c_int64),
                ("admitted", ctypes.c_int64), ("evicted", ctypes.c_int64),
                ("scratch_loads", ctypes.c_int64), ("copies", ctypes.c_int64)]

    def as_dict(self):
        return {name: getattr(self, name) for name, _ in self._fields_}


class _Append(ctypes.Structure):
    _fields_ = [("batch", ctypes.c_int32), ("max_pages_per_seq", ctypes.c_int32),
                ("num_pages", ctypes.c_int32), ("max_new", ctypes.c_int32),
                ("kv_dtype", ctypes.c_int), ("status_word", ctypes.c_void_p),
                ("stream", ctypes.c_void_p)]


_lib = None


def library_path() -> str:
    return _build.LIB


def load_library(build_if_missing: bool = False) -> ctypes.CDLL:
    """Load libatlas_attn.so; raises if it has not been built (no fallback)."""
    global _lib
    if _lib is not None:
        return _lib
    if not os.path.exists(_build.LIB):
        if not build_if_missing:
            raise ImportError(f"{_build.LIB} is missing: build it with "
                              "`python -c 'import __graft_entry__ as g; g.build()'`")
        _build.build()
    lib = ctypes.CDLL(_build.LIB)
    args = [ctypes.c_void_p] * 5 + [ctypes.c_int32] * 4 + [ctypes.c_float,
                                                           ctypes.POINTER(_Launch)]
    for name in ("atlas_attn_decode", "atlas_attn_suffix", "atlas_attn_prefill"):
        fn = getattr(lib, name)
        fn.argtypes = args
        fn.restype = ctypes.c_int
    lib.atlas_attn_workspace_size.argtypes = [ctypes.c_int] + [ctypes.c_int32] * 4 + [
        ctypes.POINTER(_Launch)]
    lib.atlas_attn_workspace_size.restype = ctypes.c_size_t
    lib.atlas_kv_append.argtypes = [ctypes.c_void_p] * 7 + [ctypes.c_int32] * 3 + [
        ctypes.POINTER(_Append)]
    lib.atlas_kv_append.restype = ctypes.c_int
    lib.atlas_attn_status_string.argtypes = [ctypes.c_int]
    lib.atlas_attn_status_string.restype = ctypes.c_char_p
    lib.atlas_attn_split_tokens.argtypes = [ctypes.c_int] + [ctypes.c_int32] * 4 + [
        ctypes.POINTER(_Launch)]
    lib.atlas_attn_split_tokens.restype = ctypes.c_int32
    lib.atlas_pool_create.argtypes = [ctypes.POINTER(_PoolConfig), ctypes.POINTER(ctypes.c_void_p)]
    lib.atlas_pool_create.restype = ctypes.c_int
    lib.atlas_pool_destroy.argtypes = [ctypes.c_void_p]
    lib.atlas_pool_destroy.restype = None
    lib.atlas_pool_plan.argtypes = [ctypes.c_void_p, ctypes.POINTER(_PoolRequest),
                                    ctypes.POINTER(PoolStats)]
    lib.atlas_pool_plan.restype = ctypes.c_int
    lib.atlas_pool_pass.argtypes = [ctypes.c_void_p, ctypes.c_int32] + [ctypes.c_void_p] * 3 + [
        ctypes.c_int32, ctypes.POINTER(ctypes.c_int32)]
    lib.atlas_pool_pass.restype = ctypes.c_int
    lib.atlas_pool_slot_of.argtypes = [ctypes.c_void_p, ctypes.c_int32]
    lib.atlas_pool_slot_of.restype = ctypes.c_int32
    lib.atlas_pool_invalidate.argtypes = [ctypes.c_void_p, ctypes.c_int32]
    lib.atlas_pool_invalidate.restype = None
    lib.atlas_pool_fill.argtypes = [ctypes.c_void_p] * 5 + [ctypes.c_int32, ctypes.c_int64,
                                                            ctypes.c_int32, ctypes.c_int32,
                                                            ctypes.c_void_p, ctypes.c_void_p]
    lib.atlas_pool_fill.restype = ctypes.c_int
    _lib = lib
    return lib


def status_string(status: int) -> str:
    return load_library().atlas_attn_status_string(status).decode()


def _ptr(t: Optional[torch.Tensor]) -> Optional[int]:
    return None if t is None else t.data_ptr()


def _launch(q, k_pages, page_table, out_dtype, out=None, lse=None, workspace=None,
            status=None, stream=None, split_tokens=0, debug_flags=0, events=None,
            window=0, softcap=0.0, sinks=None, q_lens=None, chunk_range=None,
            phase=PHASE_ALL, sm_count=0) -> _Launch:
    L = _Launch()
    L.batch, L.q_len = q.shape[0], q.shape[2]
    L.max_pages_per_seq = page_table.shape[1]
    L.num_pages = k_pages.shape[0]
    L.q_dtype = _DTYPES.get(q.dtype, -1)
    L.kv_dtype = _DTYPES.get(k_pages.dtype, -1)
    L.out_dtype = _DTYPES.get(out_dtype, -1)
    L.out = _ptr(out)
    L.lse = _ptr(lse)
    L.workspace = _ptr(workspace)
    L.workspace_bytes = 0 if workspace is None else workspace.numel() * workspace.element_size()
    L.status_word = _ptr(status)
    L.stream = stream
    L.split_tokens = split_tokens
    L.debug_flags = debug_flags
    L.events = events
    L.window = window
    L.softcap = softcap
    L.sinks = _ptr(sinks)
    L.q_lens = _ptr(q_lens)
    L.chunk_range = _ptr(chunk_range)
    L.phase = phase
    L.sm_count = sm_count
    return L


def workspace_size(kind: str, q_shape, n_q_heads, n_kv_heads, head_dim, page_tokens,
                   max_pages_per_seq, num_pages, dtype=torch.bfloat16,
                   out_dtype=None, split_tokens=0, window=0, phase=PHASE_ALL) -> int:
    """Workspace bytes a call needs (from shapes, split size, window and phase only)."""
    L = _Launch()
    L.window, L.phase = window, phase
    L.batch, L.q_len = q_shape[0], q_shape[2]
    L.max_pages_per_seq, L.num_pages = max_pages_per_seq, num_pages
    L.q_dtype = L.kv_dtype = _DTYPES.get(dtype, -1)
    L.out_dtype = _DTYPES.get(out_dtype or dtype, -1)
    L.split_tokens = split_tokens
    n = load_library().atlas_attn_workspace_size(_KINDS[kind], n_q_heads, n_kv_heads, head_dim,
                                                 page_tokens, ctypes.byref(L))
    if n == ctypes.c_size_t(-1).value:
        raise AtlasError(1, "invalid arguments for workspace_size")
    return n


def _call(kind: str, q, k_pages, v_pages, page_table, seq_lens, n_q_heads, n_kv_heads,
          head_dim, page_tokens, scale, *, out=None, out_dtype=None, lse=None,
          workspace=None, status=None, split_tokens=0, debug_flags=0, events=None,
          window=0, softcap=0.0, sinks=None, q_lens=None, chunk_range=None,
          phase=PHASE_ALL, sm_count=0):
    """``events``: optional ctypes array of three cudaEvent_t handles (see
    EventTimer) recorded around the main kernel and the merge.  ``window``,
    ``softcap`` and ``sinks`` (float32 CUDA tensor [n_q_heads]) select the score /
    mask variants; the defaults give plain causal attention.  ``q_lens`` (int32
    CUDA tensor [B]) makes the batch ragged: sequence b has q_lens[b] query rows.
    ``phase`` and ``chunk_range`` (int32 CUDA tensor [B][2]) spread one call over
    several launches sharing ``workspace`` (atlas_launch.phase).  ``sm_count`` > 0
    plans for that many SMs instead of the device's (atlas_launch.sm_count)."""
    lib = load_library()
    for name, t in (("q", q), ("k_pages", k_pages), ("v_pages", v_pages),
                    ("page_table", page_table), ("seq_lens", seq_lens)):
        if not t.is_cuda or not t.is_contiguous():
            raise ValueError(f"{name} must be a contiguous CUDA tensor")
    if page_table.dtype != torch.int32 or seq_lens.dtype != torch.int32:
        raise ValueError("page_table and seq_lens must be int32")
    if q.dim() != 4 or k_pages.dim() != 4 or v_pages.shape != k_pages.shape:
        raise ValueError("q must be [B][Hq][q_len][D] and pools [num_pages][Hkv][P][D]")
    out_dtype = out_dtype or (out.dtype if out is not None else q.dtype)
    if out is None and phase != PHASE_CHUNKS:
        out = torch.empty(q.shape, dtype=out_dtype, device=q.device)
    if chunk_range is not None and (not chunk_range.is_cuda or chunk_range.dtype != torch.int32
                                    or chunk_range.numel() != 2 * q.shape[0]
                                    or not chunk_range.is_contiguous()):
        raise ValueError("chunk_range must be a contiguous int32 CUDA tensor [batch][2]")
    if status is not None and (status.dtype != torch.int32 or status.numel() < 1):
        raise ValueError("status must be an int32 device tensor")
    if sinks is not None and (not sinks.is_cuda or sinks.dtype != torch.float32 or
                              sinks.numel() != n_q_heads or not sinks.is_contiguous()):
        raise ValueError("sinks must be a contiguous float32 CUDA tensor [n_q_heads]")
    if q_lens is not None and (not q_lens.is_cuda or q_lens.dtype != torch.int32 or
                               q_lens.numel() != q.shape[0]):
        raise ValueError("q_lens must be an int32 CUDA tensor [batch]")
    stream = torch.cuda.current_stream(q.device).cuda_stream
    L = _launch(q, k_pages, page_table, out_dtype, out, lse, None, status, stream,
                split_tokens, debug_flags,
                None if events is None else ctypes.cast(events, ctypes.c_void_p).value,
                window, softcap, sinks, q_lens, chunk_range, phase, sm_count)
    need = lib.atlas_attn_workspace_size(_KINDS[kind], n_q_heads, n_kv_heads, head_dim,
                                         page_tokens, ctypes.byref(L))
    if workspace is None and 0 < need < ctypes.c_size_t(-1).value:
        workspace = torch.empty(need, dtype=torch.uint8, device=q.device)
    L.workspace = _ptr(workspace)
    L.workspace_bytes = 0 if workspace is None else workspace.numel() * workspace.element_size()
    fn = getattr(lib, f"atlas_attn_{kind}")
    rc = fn(q.data_ptr(), k_pages.data_ptr(), v_pages.data_ptr(), page_table.data_ptr(),
            seq_lens.data_ptr(), n_q_heads, n_kv_heads, head_dim, page_tokens, float(scale),
            ctypes.byref(L))
    if rc != 0:
        raise AtlasError(rc, status_string(rc))
    return out


def split_tokens_of(kind: str, q_shape, n_q_heads, n_kv_heads, head_dim, page_tokens,
                    max_pages_per_seq, num_pages, dtype=torch.bfloat16, out_dtype=None,
                    split_tokens=0, window=0, phase=PHASE_ALL) -> int:
    """Keys per split-KV chunk of such a call (0: no chunks), atlas_attn_split_tokens."""
    L = _Launch()
    L.window, L.phase = window, phase
    L.batch, L.q_len = q_shape[0], q_shape[2]
    L.max_pages_per_seq, L.num_pages = max_pages_per_seq, num_pages
    L.q_dtype = L.kv_dtype = _DTYPES.get(dtype, -1)
    L.out_dtype = _DTYPES.get(out_dtype or dtype, -1)
    L.split_tokens = split_tokens
    n = load_library().atlas_attn_split_tokens(_KINDS[kind], n_q_heads, n_kv_heads, head_dim,
                                               page_tokens, ctypes.byref(L))
    if n < 0:
        raise AtlasError(1, "invalid arguments for split_tokens_of")
    return n


def decode(q, k_pages, v_pages, page_table, seq_lens, n_q_heads, n_kv_heads, head_dim,
           page_tokens, scale, **kw):
    """One query row per sequence (q_len == 1).  Returns out [B][Hq][1][D]."""
    return _call("decode", q, k_pages, v_pages, page_table, seq_lens, n_q_heads, n_kv_heads,
                 head_dim, page_tokens, scale, **kw)


def suffix(q, k_pages, v_pages, page_table, seq_lens, n_q_heads, n_kv_heads, head_dim,
           page_tokens, scale, **kw):
    """Queries are the last q_len positions of each sequence's K/V."""
    return _call("suffix", q, k_pages, v_pages, page_table, seq_lens, n_q_heads, n_kv_heads,
                 head_dim, page_tokens, scale, **kw)


def prefill(q, k_pages, v_pages, page_table, seq_lens, n_q_heads, n_kv_heads, head_dim,
            page_tokens, scale, **kw):
    """Causal self-attention of whole prompts (seq_lens[b] == q_len for every b)."""
    return _call("prefill", q, k_pages, v_pages, page_table, seq_lens, n_q_heads, n_kv_heads,
                 head_dim, page_tokens, scale, **kw)


def run(problem, **kw):
    """Call the entry point named by ``problem.kind`` on an inputs.Problem on the GPU."""
    fn = {"decode": decode, "suffix": suffix, "prefill": prefill}[problem.kind]
    return fn(problem.q, problem.k_pages, problem.v_pages, problem.page_table,
              problem.seq_lens, problem.n_q_heads, problem.n_kv_heads, problem.head_dim,
              problem.page_tokens, problem.scale, **kw)


def kv_append(k_new, v_new, k_pages, v_pages, page_table, seq_lens, n_new=None,
              status=None):
    """Write the new tokens' K/V rows [B][Hkv][max_new][D] of each sequence into its
    pages at positions seq_lens[b] .. seq_lens[b] + n_new[b] - 1 (atlas_kv_append).
    The pools are updated in place; seq_lens is not advanced."""
    lib = load_library()
    for name, t in (("k_new", k_new), ("v_new", v_new), ("k_pages", k_pages),
                    ("v_pages", v_pages), ("page_table", page_table), ("seq_lens", seq_lens)):
        if not t.is_cuda or not t.is_contiguous():
            raise ValueError(f"{name} must be a contiguous CUDA tensor")
    if k_new.shape != v_new.shape or k_new.dim() != 4 or k_pages.dim() != 4:
        raise ValueError("k_new/v_new must be [B][Hkv][max_new][D], pools [pages][Hkv][P][D]")
    if k_new.dtype != k_pages.dtype:
        raise ValueError("new rows and pools must share a dtype")
    A = _Append()
    A.batch, A.max_new = k_new.shape[0], k_new.shape[2]
    A.max_pages_per_seq, A.num_pages = page_table.shape[1], k_pages.shape[0]
    A.kv_dtype = _DTYPES.get(k_pages.dtype, -1)
    A.status_word = _ptr(status)
    A.stream = torch.cuda.current_stream(k_new.device).cuda_stream
    rc = lib.atlas_kv_append(k_new.data_ptr(), v_new.data_ptr(), k_pages.data_ptr(),
                             v_pages.data_ptr(), page_table.data_ptr(), seq_lens.data_ptr(),
                             _ptr(n_new), k_new.shape[1], k_new.shape[3], k_pages.shape[2],
                             ctypes.byref(A))
    if rc != 0:
        raise AtlasError(rc, status_string(rc))


class EventTimer:
    """Three torch CUDA events whose handles the library records around its main
    kernel and its merge: main_ms() and merge_ms() read them after a sync."""

    def __init__(self):
        self.ev = [torch.cuda.Event(enable_timing=True) for _ in range(3)]
        for e in self.ev:  # torch creates the CUDA event on its first record
            e.record()
        self.handles = (ctypes.c_void_p * 3)(*[e.cuda_event for e in self.ev])

    def main_ms(self) -> float:
        return self.ev[0].elapsed_time(self.ev[1])

    def merge_ms(self) -> float:
        return self.ev[1].elapsed_time(self.ev[2])


def run_host(kind: str, q, k_pages, v_pages, page_table, seq_lens, n_q_heads, n_kv_heads,
             head_dim, page_tokens, scale, *, device="cuda", out_dtype=None, host_out=None,
             **kw):
    """End-to-end call on host tensors (ideally pinned): copies the inputs to the
    device on the current stream, runs the kernels, and copies the result back.
    Returns the host output tensor (``host_out`` if given)."""
    dev = [t.to(device, non_blocking=True) for t in (q, k_pages, v_pages, page_table, seq_lens)]
    out = _call(kind, *dev, n_q_heads, n_kv_heads, head_dim, page_tokens, scale,
                out_dtype=out_dtype, **kw)
    if host_out is None:
        host_out = torch.empty(out.shape, dtype=out.dtype, pin_memory=True)
    host_out.copy_(out, non_blocking=True)
    torch.cuda.current_stream(out.device).synchronize()
    return host_out


from .pool import HotPagePool  # noqa: E402  (the pool binding uses the names above)
