"""fp64 CPU oracle for exact causal grouped-query attention over paged K/V.

TEST INFRASTRUCTURE ONLY.  The test suite, ``__graft_entry__.smoke()`` and the
benchmark's CPU-baseline leg are the only callers.  Nothing here is shared with
the CUDA library (no code, constants or helpers), and the library never calls
this package.

The arithmetic lives in ``oracle_attn.c`` (plain C, fp64, OpenMP over output
rows); this module compiles it with gcc and marshals numpy arrays into it.
Every function cites the passage it follows in the C file's header:

- ``attn``    the full-KV definition (CFR-Atlas README, "Core contract";
              ferrox-core crate index, "attention" module: the vanilla path is
              the correctness baseline).
- ``folded``  the page-by-page online-softmax fold (CFR-Atlas README, opening
              paragraph and "Core contract").
- ``state`` / ``merge``  a key-range partial state and the structured merge
              of partial states (CPUAttn README, "Operator model": split-K only
              with a structured merge).

Parity status: every function here is pinned by ``tests/test_oracle_pins.py``
(brute force at 50 digits, closed forms, invariants, and a library pin).
"""
from __future__ import annotations

import ctypes
import os
import subprocess

import numpy as np

_HERE = os.path.dirname(os.path.abspath(__file__))
_SRC = os.path.join(_HERE, "oracle_attn.c")
_LIB = os.path.join(_HERE, "_liboracle.so")
_lib = None


def build(force: bool = False) -> str:
    """Compile oracle_attn.c into _liboracle.so (gcc, -O2, OpenMP, no fast-math)."""
    if force or not os.path.exists(_LIB) or os.path.getmtime(_LIB) < os.path.getmtime(_SRC):
        tmp = _LIB + f".tmp{os.getpid()}"
        subprocess.check_call(
            ["gcc", "-O2", "-std=c11", "-fPIC", "-shared", "-fopenmp",
             "-fno-fast-math", "-ffp-contract=off", _SRC, "-o", tmp, "-lm"])
        os.replace(tmp, _LIB)
    return _LIB


def _load():
    global _lib
    if _lib is None:
        # A test that checks the pins' strength points this at a deliberately
        # broken build of oracle_attn.c; otherwise the library built here is used.
        path = os.environ.get("ATLAS_ORACLE_LIB") or build()
        lib = ctypes.CDLL(path)
        P = ctypes.c_void_p
        I = ctypes.c_int
        L = ctypes.c_int64
        Dd = ctypes.c_double
        common = [P, P, P, P, P, I, I, I, I, I, I, I, I, Dd, I, Dd]
        for name in ("oracle_attn", "oracle_folded"):
            fn = getattr(lib, name)
            fn.argtypes = common + [P, P, P, L, P, P]
            fn.restype = I
        lib.oracle_kv_append.argtypes = [P] * 7 + [I] * 7
        lib.oracle_kv_append.restype = I
        lib.oracle_state.argtypes = common + [L, L, L, P, P, P]
        lib.oracle_state.restype = I
        lib.oracle_merge.argtypes = [I, I, P, P, P, P, P]
        lib.oracle_merge.restype = I
        lib.oracle_num_threads.argtypes = []
        lib.oracle_num_threads.restype = I
        _lib = lib
    return _lib


class OracleError(RuntimeError):
    pass


_ERRORS = {1: "bad argument", 2: "row without visible keys or context beyond the page table",
           3: "page id out of range", 4: "out of memory"}


def _f32(x) -> np.ndarray:
    if hasattr(x, "detach"):  # torch tensor: widen exactly to fp32 on the CPU
        x = x.detach().to("cpu").float().numpy()
    return np.ascontiguousarray(x, dtype=np.float32)


def _i32(x) -> np.ndarray:
    if hasattr(x, "detach"):
        x = x.detach().to("cpu").numpy()
    return np.ascontiguousarray(x, dtype=np.int32)


def _ptr(a: np.ndarray):
    return a.ctypes.data_as(ctypes.c_void_p)


def num_threads() -> int:
    """OpenMP threads the oracle runs with (OMP_NUM_THREADS or all cores)."""
    return _load().oracle_num_threads()


def _prepare(q, k_pages, v_pages, page_table, seq_lens, n_q_heads, n_kv_heads):
    q = _f32(q)
    k = _f32(k_pages)
    v = _f32(v_pages)
    table = _i32(page_table)
    lens = _i32(seq_lens)
    if q.ndim != 4 or k.ndim != 4 or k.shape != v.shape or table.ndim != 2:
        raise OracleError("expected q[B][Hq][q_len][D], pools[num_pages][Hkv][P][D], table[B][max_pages]")
    B, Hq, q_len, D = q.shape
    num_pages, Hkv, P, Dk = k.shape
    if Hq != n_q_heads or Hkv != n_kv_heads or Dk != D or table.shape[0] != B or lens.shape != (B,):
        raise OracleError("inconsistent shapes")
    dims = (B, Hq, Hkv, D, P, table.shape[1], num_pages, q_len)
    return q, k, v, table, lens, dims


def _run(name, q, k_pages, v_pages, page_table, seq_lens, n_q_heads, n_kv_heads, scale,
         rows=None, want_lse=False, window=0, softcap=0.0, sinks=None, q_lens=None):
    lib = _load()
    q, k, v, table, lens, dims = _prepare(q, k_pages, v_pages, page_table, seq_lens,
                                          n_q_heads, n_kv_heads)
    B, Hq, Hkv, D, P, max_pages, num_pages, q_len = dims
    sinks_arr = None if sinks is None else _f32(sinks)
    if sinks_arr is not None and sinks_arr.shape != (Hq,):
        raise OracleError("sinks must hold one logit per q head")
    qlen_arr = None if q_lens is None else _i32(q_lens)
    if qlen_arr is not None and qlen_arr.shape != (B,):
        raise OracleError("q_lens must hold one count per sequence")
    if rows is None:
        n_rows = B * Hq * q_len
        rows_arr = None
    else:
        rows_arr = np.ascontiguousarray(rows, dtype=np.int64)
        n_rows = rows_arr.size
    out = np.empty((n_rows, D), dtype=np.float64)
    lse = np.empty(n_rows, dtype=np.float64) if want_lse else None
    rc = getattr(lib, name)(
        _ptr(q), _ptr(k), _ptr(v), _ptr(table), _ptr(lens), *dims, float(scale),
        int(window), float(softcap), _ptr(sinks_arr) if sinks_arr is not None else None,
        _ptr(qlen_arr) if qlen_arr is not None else None,
        _ptr(rows_arr) if rows_arr is not None else None, n_rows,
        _ptr(out), _ptr(lse) if lse is not None else None)
    if rc:
        raise OracleError(f"{name}: {_ERRORS.get(rc, rc)}")
    if rows is None:
        out = out.reshape(B, Hq, q_len, D)
        if lse is not None:
            lse = lse.reshape(B, Hq, q_len)
    return (out, lse) if want_lse else out


def attn(q, k_pages, v_pages, page_table, seq_lens, n_q_heads, n_kv_heads, scale,
         rows=None, want_lse=False, window=0, softcap=0.0, sinks=None, q_lens=None):
    """Full-KV causal GQA attention in fp64.

    q[B][Hq][q_len][D]; pools [num_pages][Hkv][P][D]; page_table[B][max_pages];
    seq_lens[B].  Query row i of sequence b sits at position seq_lens[b] - q_len + i
    and sees keys 0..that position (only the last ``window`` of them when window > 0);
    ``softcap`` c > 0 maps each scaled score s to c tanh(s / c); ``sinks`` (one logit
    per q head) adds exp(sink) to the softmax denominator.  ``q_lens`` (ragged query
    counts, <= q_len) makes row i of sequence b a query only when i < q_lens[b], at
    position seq_lens[b] - q_lens[b] + i (padding rows: 0, lse NaN).  ``rows`` (flat indices
    (b*Hq+h)*q_len+i) restricts the output to those rows, returned as [len(rows)][D].
    """
    return _run("oracle_attn", q, k_pages, v_pages, page_table, seq_lens, n_q_heads,
                n_kv_heads, scale, rows, want_lse, window, softcap, sinks, q_lens)


def folded(q, k_pages, v_pages, page_table, seq_lens, n_q_heads, n_kv_heads, scale,
           rows=None, want_lse=False, window=0, softcap=0.0, sinks=None, q_lens=None):
    """The same result reached by folding one page at a time into (m, l, acc)."""
    return _run("oracle_folded", q, k_pages, v_pages, page_table, seq_lens, n_q_heads,
                n_kv_heads, scale, rows, want_lse, window, softcap, sinks, q_lens)


def state(q, k_pages, v_pages, page_table, seq_lens, n_q_heads, n_kv_heads, scale,
          row, t_begin, t_end, window=0, softcap=0.0):
    """(m, l, acc) of flat row ``row`` over its visible keys in [t_begin, t_end)."""
    lib = _load()
    q, k, v, table, lens, dims = _prepare(q, k_pages, v_pages, page_table, seq_lens,
                                          n_q_heads, n_kv_heads)
    D = dims[3]
    m = np.zeros(1)
    l = np.zeros(1)
    acc = np.zeros(D)
    rc = lib.oracle_state(_ptr(q), _ptr(k), _ptr(v), _ptr(table), _ptr(lens), *dims,
                          float(scale), int(window), float(softcap), int(row), int(t_begin),
                          int(t_end), _ptr(m), _ptr(l), _ptr(acc))
    if rc:
        raise OracleError(f"oracle_state: {_ERRORS.get(rc, rc)}")
    return float(m[0]), float(l[0]), acc


def merge(ms, ls, accs):
    """Combine partial states (m_s, l_s, acc_s) into (o, lse)."""
    lib = _load()
    m = np.ascontiguousarray(ms, dtype=np.float64)
    l = np.ascontiguousarray(ls, dtype=np.float64)
    acc = np.ascontiguousarray(accs, dtype=np.float64)
    S, D = acc.shape
    out = np.empty(D)
    lse = np.empty(1)
    rc = lib.oracle_merge(S, D, _ptr(m), _ptr(l), _ptr(acc), _ptr(out), _ptr(lse))
    if rc:
        raise OracleError(f"oracle_merge: {_ERRORS.get(rc, rc)}")
    return out, float(lse[0])


def kv_append(k_new, v_new, k_pages, v_pages, page_table, seq_lens, n_new=None):
    """Write new K/V rows [B][Hkv][max_new][D] of each sequence to the page slots of
    positions seq_lens[b] .. seq_lens[b] + n_new[b] - 1.  Returns new float64-exact
    float32 pools (the inputs are not modified)."""
    lib = _load()
    kn, vn = _f32(k_new), _f32(v_new)
    kp, vp = _f32(k_pages).copy(), _f32(v_pages).copy()
    table, lens = _i32(page_table), _i32(seq_lens)
    nn = None if n_new is None else _i32(n_new)
    B, Hkv, max_new, D = kn.shape
    num_pages, _, P, _ = kp.shape
    rc = lib.oracle_kv_append(_ptr(kn), _ptr(vn), _ptr(kp), _ptr(vp), _ptr(table), _ptr(lens),
                              _ptr(nn) if nn is not None else None, B, Hkv, max_new, D, P,
                              table.shape[1], num_pages)
    if rc:
        raise OracleError(f"oracle_kv_append: {_ERRORS.get(rc, rc)}")
    return kp, vp
