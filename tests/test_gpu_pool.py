"""GPU checks of the bounded hot-page pool: the fill kernel copies pages exactly,
and a decode served from a pool smaller than the context equals the decode over a
fully resident pool bit for bit (hence the oracle within tolerance), whatever the
pool held before, the budget, the KeepRecent window or the admission switch."""
import numpy as np
import pytest
import torch

import exact_causal_gqa_gb300 as atlas
from exact_causal_gqa_gb300 import inputs
from tests.gpu_helpers import assert_parity, oracle_rows

pytestmark = pytest.mark.gpu


def host_problem(dtype="bf16", B=4, Hq=16, Hkv=4, D=128, P=16, lens=(700, 2100, 64, 1333),
                 seed=11, out_dtype=None):
    prob = inputs.make("decode", B, Hq, Hkv, D, P, list(lens), q_len=1, dtype=dtype,
                       out_dtype=out_dtype or dtype, seed=seed, device="cpu", extra_pages=5)
    return prob


def to_device(prob):
    return inputs.Problem(**{k: (v.cuda() if torch.is_tensor(v) else v)
                             for k, v in vars(prob).items()})


def pinned(t):
    return t.contiguous().pin_memory()


def test_fill_copies_pages_exactly():
    torch.manual_seed(0)
    host_k = pinned(torch.randn(40, 4, 16, 128).to(torch.bfloat16))
    host_v = pinned(torch.randn(40, 4, 16, 128).to(torch.bfloat16))
    pool = atlas.HotPagePool(host_k, host_v, hot_slots=6, scratch_slots=4)
    pool.k_slots.zero_()
    pool.v_slots.zero_()
    pairs = torch.tensor([[7, 0], [39, 9], [0, 3], [7, 5], [22, 8]], dtype=torch.int32)
    status = torch.zeros(1, dtype=torch.int32, device="cuda")
    pool.fill(pairs.cuda(), status)
    torch.cuda.synchronize()
    for hp, s in pairs.tolist():
        assert torch.equal(pool.k_slots[s].cpu(), host_k[hp])
        assert torch.equal(pool.v_slots[s].cpu(), host_v[hp])
    untouched = [s for s in range(10) if s not in pairs[:, 1].tolist()]
    assert pool.k_slots[untouched].abs().sum().item() == 0
    assert status.item() == 0
    # a pair outside the host tier or the slots is skipped and flagged
    bad = torch.tensor([[40, 1], [3, 10], [-1, 2], [5, 1]], dtype=torch.int32)
    pool.fill(bad.cuda(), status)
    torch.cuda.synchronize()
    assert status.item() & atlas.DEV_BAD_PAGE
    assert torch.equal(pool.k_slots[1].cpu(), host_k[5])
    assert pool.k_slots[2].abs().sum().item() == 0
    pool.close()


def reference(prob_dev, out_dtype, split_tokens):
    lse = torch.empty(prob_dev.q.shape[:3], dtype=torch.float32, device="cuda")
    out = atlas.run(prob_dev, out_dtype=out_dtype, lse=lse, split_tokens=split_tokens)
    return out, lse


@pytest.mark.parametrize("dtype,out_dtype", [("bf16", torch.float32), ("bf16", torch.bfloat16),
                                             ("f32", torch.float32)])
def test_pooled_decode_is_bit_identical_to_resident_decode(dtype, out_dtype):
    prob = host_problem(dtype=dtype, D=128 if dtype == "bf16" else 64)
    dev = to_device(prob)
    split = 256
    ref, ref_lse = reference(dev, out_dtype, split)
    host_k, host_v = pinned(prob.k_pages), pinned(prob.v_pages)
    table, lens = prob.page_table.contiguous(), prob.seq_lens.contiguous()
    chunk_pages = split // prob.page_tokens + 1
    pool = atlas.HotPagePool(host_k, host_v, hot_slots=30, scratch_slots=2 * chunk_pages)
    seen_passes = set()
    for keep, admit in ((512, True), (512, True), (-1, True), (0, True), (-1, False),
                        (128, True), (-1, True)):
        lse = torch.empty_like(ref_lse)
        out, st = pool.decode(dev.q, table, lens, prob.n_q_heads, prob.scale,
                              keep_recent_tokens=keep, admit=admit, out_dtype=out_dtype,
                              lse=lse, split_tokens=split)
        torch.cuda.synchronize()
        seen_passes.add(st.passes)
        assert torch.equal(out, ref), (keep, admit, st.as_dict())
        assert torch.equal(lse, ref_lse)
    assert max(seen_passes) > 1  # the context did not fit: several passes were needed
    # a rewritten host page: invalidate, then the pool serves the new contents
    hot = [hp for hp in table.flatten().tolist() if pool.slot_of(hp) >= 0]
    assert hot
    hp = hot[0]
    host_k[hp].copy_(host_k[hp] * 0.5)
    dev.k_pages[hp].copy_(host_k[hp].cuda())
    pool.invalidate(hp)
    ref2, _ = reference(dev, out_dtype, split)
    out, _ = pool.decode(dev.q, table, lens, prob.n_q_heads, prob.scale, out_dtype=out_dtype,
                         split_tokens=split)
    torch.cuda.synchronize()
    assert torch.equal(out, ref2)
    pool.close()


def test_pooled_decode_matches_the_oracle_with_automatic_splits():
    prob = host_problem(lens=(5000, 300, 2600, 9000), seed=5)
    dev = to_device(prob)
    pool = atlas.HotPagePool(pinned(prob.k_pages), pinned(prob.v_pages), hot_slots=64,
                             scratch_slots=200)
    for _ in range(2):
        out, st = pool.decode(dev.q, prob.page_table, prob.seq_lens, prob.n_q_heads,
                              prob.scale, keep_recent_tokens=1024, out_dtype=torch.float32)
        torch.cuda.synchronize()
        assert_parity(prob, out, oracle_rows(prob), "pooled decode")
    assert st.hits > 0 and st.passes > 1
    ref = atlas.run(dev, out_dtype=torch.float32)
    assert torch.equal(out, ref)
    pool.close()


def test_pooled_decode_on_the_tensor_core_path():
    # G = 32 query heads per kv head: the decode takes the tcgen05 path, whose
    # chunked form the passes use.  The passes keep fixed chunks (their split size
    # for the chunked phases); a resident call with that split size gives the same
    # bits (an automatic resident call cuts each sequence into equal splits instead,
    # equal within the tolerance, not bitwise).
    prob = host_problem(B=2, Hq=32, Hkv=1, lens=(3000, 1500), seed=3)
    dev = to_device(prob)
    chunk = atlas.split_tokens_of("decode", dev.q.shape, prob.n_q_heads, prob.n_kv_heads,
                                  prob.head_dim, prob.page_tokens, prob.max_pages,
                                  prob.num_pages, dev.q.dtype, torch.float32,
                                  phase=atlas.PHASE_CHUNKS)
    ref = atlas.run(dev, out_dtype=torch.float32, split_tokens=chunk)
    pool = atlas.HotPagePool(pinned(prob.k_pages), pinned(prob.v_pages), hot_slots=16,
                             scratch_slots=80)
    out, st = pool.decode(dev.q, prob.page_table, prob.seq_lens, prob.n_q_heads, prob.scale,
                          keep_recent_tokens=256, out_dtype=torch.float32)
    torch.cuda.synchronize()
    assert torch.equal(out, ref)
    assert_parity(prob, out, oracle_rows(prob), "pooled tensor-core decode")
    pool.close()


def test_device_host_tier_and_shared_pages():
    # two sequences reading the same pages (a shared prefix) from a device-memory tier
    prob = host_problem(B=2, lens=(900, 900), seed=8)
    prob.page_table[1] = prob.page_table[0]
    dev = to_device(prob)
    ref = atlas.run(dev, out_dtype=torch.float32, split_tokens=128)
    pool = atlas.HotPagePool(dev.k_pages, dev.v_pages, hot_slots=10, scratch_slots=20)
    out, st = pool.decode(dev.q, prob.page_table, prob.seq_lens, prob.n_q_heads, prob.scale,
                          out_dtype=torch.float32, split_tokens=128)
    torch.cuda.synchronize()
    assert torch.equal(out, ref)
    assert st.pages == (900 + 15) // 16
    pool.close()


def test_pageable_host_tier_is_refused():
    k = torch.zeros(4, 1, 16, 64)
    with pytest.raises(ValueError):
        atlas.HotPagePool(k, k.clone(), 2, 2)
    pool = atlas.HotPagePool(k.pin_memory(), k.pin_memory(), 2, 2)
    pool.host_k = k  # bypass the binding's check: the library itself refuses it
    with pytest.raises(atlas.AtlasError):
        pool.fill(torch.tensor([[0, 0]], dtype=torch.int32, device="cuda"))
    pool.close()
