"""CPU checks of the bounded hot-page pool's planner (host code, no GPU).

The plain model in oracle/pool_model.py is pinned by hand-worked traces
(tests/golden/pool_traces.json); the native planner in libatlas_attn.so must
reproduce those traces and agree with the model, pass by pass, on random traces.
"""
import ctypes
import json
import os
import random

import numpy as np
import pytest

import exact_causal_gqa_gb300 as atlas
from exact_causal_gqa_gb300 import _build
from oracle.pool_model import PoolModel

HERE = os.path.dirname(os.path.abspath(__file__))
TRACES = json.load(open(os.path.join(HERE, "golden", "pool_traces.json")))


@pytest.fixture(scope="module")
def lib():
    _build.build()
    return atlas.load_library()


class Native:
    """The library's planner through its C ABI (atlas_pool_*)."""

    def __init__(self, lib, hot, scratch, P, host_pages):
        self.lib, self.H, self.C, self.P = lib, hot, scratch, P
        cfg = atlas._PoolConfig(hot, scratch, P, host_pages)
        self.h = ctypes.c_void_p()
        assert lib.atlas_pool_create(ctypes.byref(cfg), ctypes.byref(self.h)) == 0

    def __del__(self):
        self.lib.atlas_pool_destroy(self.h)

    def plan(self, table, seq_lens, chunk, keep_recent=-1, admit=True):
        B = len(table)
        MP = max(len(r) for r in table)
        tab = np.zeros((B, MP), dtype=np.int32)
        for b, r in enumerate(table):
            tab[b, :len(r)] = r
        lens = np.asarray(seq_lens, dtype=np.int32)
        req = atlas._PoolRequest(B, MP, tab.ctypes.data, lens.ctypes.data, chunk, keep_recent,
                                 1 if admit else 0)
        st = atlas.PoolStats()
        rc = self.lib.atlas_pool_plan(self.h, ctypes.byref(req), ctypes.byref(st))
        if rc != 0:
            return rc, None, None
        passes = []
        cap = self.H + self.C
        for k in range(st.passes):
            t = np.zeros((B, MP), dtype=np.int32)
            rg = np.zeros((B, 2), dtype=np.int32)
            cp = np.zeros((cap, 2), dtype=np.int32)
            n = ctypes.c_int32()
            assert self.lib.atlas_pool_pass(self.h, k, t.ctypes.data, rg.ctypes.data,
                                            cp.ctypes.data, cap, ctypes.byref(n)) == 0
            passes.append((t, rg, [tuple(x) for x in cp[:n.value].tolist()]))
        return 0, st.as_dict(), passes

    def slot_of(self, page):
        return self.lib.atlas_pool_slot_of(self.h, page)

    def invalidate(self, page):
        self.lib.atlas_pool_invalidate(self.h, page)


def reads_of(table, ranges, seq_lens, P, chunk):
    """(b, j) -> slot for the pages a native pass reads: those of its chunk range."""
    reads = {}
    for b, (lo, hi) in enumerate(ranges.tolist()):
        for c in range(lo, hi):
            t0, t1 = c * chunk, min((c + 1) * chunk, seq_lens[b])
            for j in range(t0 // P, (t1 - 1) // P + 1):
                reads[(b, j)] = int(table[b, j])
    return reads


def check_call_against_golden(passes_reads, passes_ranges, passes_copies, stats, call):
    assert stats == call["stats"], call["derivation"]
    assert len(passes_reads) == len(call["passes"])
    for got_r, got_g, got_c, exp in zip(passes_reads, passes_ranges, passes_copies,
                                        call["passes"]):
        assert got_r == {(b, j): s for b, j, s in exp["reads"]}, call["derivation"]
        assert got_g == {b: (lo, hi) for b, lo, hi in exp["ranges"]}, call["derivation"]
        assert sorted(got_c) == sorted(tuple(c) for c in exp["copies"]), call["derivation"]


def test_model_reproduces_the_hand_worked_traces():
    cfg = TRACES["config"]
    m = PoolModel(cfg["hot_slots"], cfg["scratch_slots"], cfg["page_tokens"])
    for call in TRACES["calls"]:
        passes, stats = m.plan(call["table"], call["seq_lens"], call["chunk"],
                               call["keep_recent"], call["admit"])
        check_call_against_golden([dict(p.table) for p in passes],
                                  [dict(p.ranges) for p in passes],
                                  [p.copies for p in passes], stats, call)
        for page, slot in call["resident"].items():
            assert m.slot_of(int(page)) == slot, call["derivation"]


def test_native_planner_reproduces_the_hand_worked_traces(lib):
    cfg = TRACES["config"]
    P = cfg["page_tokens"]
    n = Native(lib, cfg["hot_slots"], cfg["scratch_slots"], P, cfg["host_pages"])
    for call in TRACES["calls"]:
        rc, stats, passes = n.plan(call["table"], call["seq_lens"], call["chunk"],
                                   call["keep_recent"], call["admit"])
        assert rc == 0
        reads = [reads_of(t, rg, call["seq_lens"], P, call["chunk"]) for t, rg, _ in passes]
        ranges = [{b: (int(lo), int(hi)) for b, (lo, hi) in enumerate(rg.tolist()) if hi > lo}
                  for _, rg, _ in passes]
        check_call_against_golden(reads, ranges, [c for _, _, c in passes], stats, call)
        for page, slot in call["resident"].items():
            assert n.slot_of(int(page)) == slot, call["derivation"]


def random_call(rng, host_pages, P, max_b=4, max_pages=9):
    B = rng.randint(1, max_b)
    table, lens = [], []
    for _ in range(B):
        L = rng.randint(1, max_pages * P)
        np_ = (L + P - 1) // P
        # pages drawn with repeats across sequences (shared prefixes / pages)
        table.append([rng.randrange(host_pages) for _ in range(np_)])
        lens.append(L)
    return table, lens


@pytest.mark.parametrize("seed", range(12))
def test_native_planner_agrees_with_the_model(lib, seed):
    rng = random.Random(seed)
    P = rng.choice([8, 16])
    H = rng.randint(0, 6)
    host_pages = rng.randint(4, 24)
    chunk = rng.choice([P, 2 * P, 3 * P, P + 8, 40])
    per_chunk = (chunk + P - 2) // P + 1  # pages a chunk can span
    C = rng.randint(per_chunk, per_chunk + 3)
    m = PoolModel(H, C, P)
    n = Native(lib, H, C, P, host_pages)
    for call_no in range(25):
        if rng.random() < 0.15:
            page = rng.randrange(host_pages)
            m.invalidate(page)
            n.invalidate(page)
        table, lens = random_call(rng, host_pages, P)
        keep = rng.choice([-1, 0, 1, P, 3 * P, 1000])
        admit = rng.random() < 0.8
        mp, ms = m.plan(table, lens, chunk, keep, admit)
        rc, ns, npasses = n.plan(table, lens, chunk, keep, admit)
        assert rc == 0
        assert ns == ms, (seed, call_no)
        assert len(npasses) == len(mp)
        for (t, rg, cp), ps in zip(npasses, mp):
            assert reads_of(t, rg, lens, P, chunk) == dict(ps.table), (seed, call_no)
            got = {b: (int(lo), int(hi)) for b, (lo, hi) in enumerate(rg.tolist()) if hi > lo}
            assert got == dict(ps.ranges)
            assert cp == ps.copies  # same order: scratch copies, then admissions, per chunk
        for page in range(host_pages):
            assert n.slot_of(page) == m.slot_of(page), (seed, call_no, page)


@pytest.mark.parametrize("seed", range(6))
def test_plan_invariants(lib, seed):
    """Whatever the policy: each pass copies at most scratch_slots pages into scratch,
    every page a pass reads sits in a hot slot that holds it or was copied into its
    scratch slot by that pass, chunks are covered exactly once, in order."""
    rng = random.Random(100 + seed)
    P, H, C, host_pages, chunk = 16, rng.randint(0, 5), 3, 30, 32
    n = Native(lib, H, C, P, host_pages)
    resident = {}  # host page -> hot slot, tracked from the copies
    for _ in range(20):
        table, lens = random_call(rng, host_pages, P, max_b=5, max_pages=8)
        rc, st, passes = n.plan(table, lens, chunk, rng.choice([-1, 0, 2 * P]), True)
        assert rc == 0
        covered = {b: [] for b in range(len(lens))}
        for t, rg, cp in passes:
            scratch = [(hp, s) for hp, s in cp if s >= H]
            assert len(scratch) <= C
            assert len({s for _, s in scratch}) == len(scratch)
            for hp, s in cp:
                if s < H:
                    for k in [k for k, v in resident.items() if v == s]:
                        del resident[k]
                    resident[hp] = s
            here = set(cp)  # a page may be copied twice in a pass: scratch, then admitted
            for (b, j), s in reads_of(t, rg, lens, P, chunk).items():
                hp = table[b][j]
                assert (s < H and resident.get(hp) == s) or (s >= H and (hp, s) in here)
            for b, (lo, hi) in enumerate(rg.tolist()):
                covered[b] += list(range(lo, hi))
        for b, L in enumerate(lens):
            assert covered[b] == list(range((L + chunk - 1) // chunk))
        assert st["copies"] == sum(len(cp) for _, _, cp in passes)
        for page in range(host_pages):
            assert n.slot_of(page) == resident.get(page, -1)


def test_invalid_requests_leave_the_pool_unchanged(lib):
    P, H, C = 8, 2, 2
    n = Native(lib, H, C, P, 10)
    m = PoolModel(H, C, P)
    assert n.plan([[1, 2]], [16], 16, -1, True)[0] == 0
    m.plan([[1, 2]], [16], 16, -1, True)
    bad = [
        ([[1, 2, 3]], [24], 24),   # a chunk of 3 pages cannot fit 2 scratch slots
        ([[1, 12]], [16], 16),     # host page outside [0, host_pages)
        ([[1, 2]], [17], 16),      # seq_len past max_pages * P
        ([[1, 2]], [0], 16),       # empty sequence
        ([[1, 2]], [16], 0),       # no chunk size
    ]
    for table, lens, chunk in bad:
        assert n.plan(table, lens, chunk, -1, True)[0] == 1
        for page in range(10):
            assert n.slot_of(page) == m.slot_of(page)
    # the failed plans left no trace: the next plan matches the model's
    _, ms = m.plan([[3, 4]], [16], 16, -1, True)
    rc, ns, _ = n.plan([[3, 4]], [16], 16, -1, True)
    assert rc == 0 and ns == ms


def test_pool_config_checks(lib):
    h = ctypes.c_void_p()
    for hot, scratch, P, pages in ((-1, 1, 16, 4), (1, 0, 16, 4), (1, 1, 12, 4), (1, 1, 256, 4),
                                   (1, 1, 16, 0)):
        cfg = atlas._PoolConfig(hot, scratch, P, pages)
        assert lib.atlas_pool_create(ctypes.byref(cfg), ctypes.byref(h)) == 1
    assert lib.atlas_pool_slot_of(None, 0) == -1
