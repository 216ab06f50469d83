"""Test-side data movement: logical K/V -> pages, and back.

Independent of both the oracle and the CUDA library: it only copies rows, so
pins can state expected values on logical (unpaged) arrays and still exercise
the page-table indexing of whatever consumes the pages.
"""
import numpy as np


def page_kv(k_log, v_log, lens, P, seed=0, pad_page=0, extra_pages=0, poison=True):
    """Scatter logical K/V [B][Hkv][Lmax][D] into a shuffled pool of P-token pages.

    Returns (k_pages, v_pages, page_table): pools [num_pages][Hkv][P][D] float32 and
    page_table [B][max_pages] int32.  Tail slots and unused pages hold NaN.
    """
    k_log = np.asarray(k_log, dtype=np.float32)
    v_log = np.asarray(v_log, dtype=np.float32)
    B, Hkv, _, D = k_log.shape
    n_pages = [(int(L) + P - 1) // P for L in lens]
    num = max(1, sum(n_pages) + extra_pages)
    perm = np.random.default_rng(seed).permutation(num)
    fill = np.nan if poison else 0.0
    k_pool = np.full((num, Hkv, P, D), fill, dtype=np.float32)
    v_pool = np.full((num, Hkv, P, D), fill, dtype=np.float32)
    table = np.full((B, max(1, max(n_pages))), pad_page, dtype=np.int32)
    c = 0
    for b, L in enumerate(lens):
        for p in range(n_pages[b]):
            phys = int(perm[c])
            c += 1
            table[b, p] = phys
            t0, t1 = p * P, min(int(L), p * P + P)
            k_pool[phys, :, : t1 - t0] = k_log[b, :, t0:t1]
            v_pool[phys, :, : t1 - t0] = v_log[b, :, t0:t1]
    return k_pool, v_pool, table


def gather_kv(k_pages, v_pages, table, lens):
    """Inverse of page_kv: logical K/V [B][Hkv][max(lens)][D] (padding zero)."""
    k_pages = np.asarray(k_pages, dtype=np.float32)
    v_pages = np.asarray(v_pages, dtype=np.float32)
    table = np.asarray(table)
    num, Hkv, P, D = k_pages.shape
    B = len(lens)
    Lmax = max(int(x) for x in lens)
    k = np.zeros((B, Hkv, Lmax, D), dtype=np.float32)
    v = np.zeros((B, Hkv, Lmax, D), dtype=np.float32)
    for b, L in enumerate(lens):
        for t in range(int(L)):
            phys = table[b, t // P]
            k[b, :, t] = k_pages[phys, :, t % P]
            v[b, :, t] = v_pages[phys, :, t % P]
    return k, v
