"""The paged KV append and ragged query counts (chunked prefill), against the
fp64 oracle on the same host bytes.  Needs a GB300."""
import numpy as np
import pytest
import torch

import exact_causal_gqa_gb300 as atlas
import oracle
from exact_causal_gqa_gb300 import inputs
from tests.gpu_helpers import assert_parity, flat_rows, oracle_rows, run_gpu

pytestmark = pytest.mark.gpu
DEV = "cuda"


def grown_problem(dtype, P, old, new, seed, Hq=8, Hkv=2, D=128):
    """A problem whose pages are sized for old + new tokens; returns it with the
    new rows [B][Hkv][max_new][D] and the pools as they were before the append."""
    total = [o + n for o, n in zip(old, new)]
    prob = inputs.make("decode", len(old), Hq, Hkv, D, P, total, dtype=dtype, seed=seed,
                       poison=False)
    tdt = prob.k_pages.dtype
    max_new = max(max(new), 1)
    g = torch.Generator().manual_seed(seed + 1)
    k_new = torch.randn((len(old), Hkv, max_new, D), generator=g).to(tdt)
    v_new = torch.randn((len(old), Hkv, max_new, D), generator=g).to(tdt)
    return prob, k_new, v_new


@pytest.mark.parametrize("dtype,P,D", [("bf16", 16, 128), ("bf16", 64, 128), ("f32", 16, 64),
                                       ("bf16", 128, 64)])
def test_append_matches_oracle_bitwise(dtype, P, D):
    old, new = [5, 130, 0, 63], [11, 1, 40, 2]
    prob, k_new, v_new = grown_problem(dtype, P, old, new, 50 + P, D=D)
    dev = prob.to(DEV)
    seq_old = torch.tensor(old, dtype=torch.int32)
    n_new = torch.tensor(new, dtype=torch.int32)
    status = torch.zeros(1, dtype=torch.int32, device=DEV)
    atlas.kv_append(k_new.to(DEV), v_new.to(DEV), dev.k_pages, dev.v_pages, dev.page_table,
                    seq_old.to(DEV), n_new.to(DEV), status=status)
    torch.cuda.synchronize()
    assert int(status.item()) == 0
    kp, vp = oracle.kv_append(k_new, v_new, prob.k_pages, prob.v_pages, prob.page_table,
                              seq_old, n_new)
    assert np.array_equal(dev.k_pages.float().cpu().numpy(), kp)
    assert np.array_equal(dev.v_pages.float().cpu().numpy(), vp)


def test_append_bad_page_is_flagged_and_skipped():
    old, new = [10, 20], [8, 8]
    prob, k_new, v_new = grown_problem("bf16", 16, old, new, 60)
    prob.page_table[0, 1] = prob.num_pages + 3       # positions 16.. of sequence 0
    dev = prob.to(DEV)
    before = dev.k_pages.clone()
    status = torch.zeros(1, dtype=torch.int32, device=DEV)
    atlas.kv_append(k_new.to(DEV), v_new.to(DEV), dev.k_pages, dev.v_pages, dev.page_table,
                    torch.tensor(old, dtype=torch.int32, device=DEV),
                    torch.tensor(new, dtype=torch.int32, device=DEV), status=status)
    torch.cuda.synchronize()
    assert int(status.item()) & atlas.DEV_BAD_PAGE
    # sequence 1 was written in full
    good = prob.page_table[1].long()
    assert not torch.equal(before[good[1]], dev.k_pages[good[1]])


def test_append_then_decode_is_a_serving_step():
    old, new = [300, 1000, 17], [1, 1, 1]
    prob, k_new, v_new = grown_problem("bf16", 16, old, new, 61, Hq=16, Hkv=4)
    dev = prob.to(DEV)
    seq_old = torch.tensor(old, dtype=torch.int32, device=DEV)
    atlas.kv_append(k_new.to(DEV), v_new.to(DEV), dev.k_pages, dev.v_pages, dev.page_table,
                    seq_old, None)
    out = run_gpu(dev, out_dtype=torch.float32)     # dev.seq_lens = old + new
    torch.cuda.synchronize()
    kp, vp = oracle.kv_append(k_new, v_new, prob.k_pages, prob.v_pages, prob.page_table,
                              torch.tensor(old, dtype=torch.int32), None)
    grown = inputs.Problem(**{**prob.__dict__, "k_pages": torch.from_numpy(kp),
                              "v_pages": torch.from_numpy(vp)})
    assert_parity(grown, out, oracle_rows(grown), "append + decode")


RAGGED = [
    # (kind, B, Hq, Hkv, P, q_len, seq_lens, q_lens, call kwargs)
    ("suffix", 3, 32, 4, 32, 16, [400, 90, 1000], [16, 5, 1], {}),
    ("suffix", 3, 32, 4, 32, 16, [400, 90, 1000], [16, 5, 0], dict(split_tokens=128)),
    ("suffix", 2, 8, 4, 16, 4, [300, 61], [4, 2], {}),                 # split (mma.sync) path
    ("prefill", 3, 8, 2, 64, 512, [512, 300, 17], [512, 300, 17],
     dict(debug_flags=atlas.DEBUG_TC_DIRECT)),
    ("prefill", 3, 8, 2, 64, 512, [512, 300, 17], [512, 300, 17], dict(split_tokens=256)),
    ("prefill", 2, 6, 2, 16, 200, [200, 129], [200, 129], dict(debug_flags=atlas.DEBUG_TC_DIRECT)),
]


@pytest.mark.parametrize("kind,B,Hq,Hkv,P,q_len,lens,q_lens,kw", RAGGED)
def test_ragged_batches(kind, B, Hq, Hkv, P, q_len, lens, q_lens, kw):
    prob = inputs.make("suffix", B, Hq, Hkv, 128, P, lens, q_len=q_len, seed=70 + q_len)
    prob.kind = kind
    ref, ref_lse = oracle_rows(prob, want_lse=True, q_lens=np.int32(q_lens))
    dev = prob.to(DEV)
    ql = torch.tensor(q_lens, dtype=torch.int32, device=DEV)
    sentinel = 12345.0
    out = torch.full(prob.q.shape, sentinel, dtype=torch.float32, device=DEV)
    lse = torch.full((flat_rows(prob),), sentinel, dtype=torch.float32, device=DEV)
    status = torch.zeros(1, dtype=torch.int32, device=DEV)
    run_gpu(dev, out=out, out_dtype=torch.float32, lse=lse, status=status, q_lens=ql, **kw)
    torch.cuda.synchronize()
    assert int(status.item()) == 0
    got = out.cpu()
    for b in range(B):
        qn = q_lens[b]
        if qn:
            assert_parity(prob, got[b, :, :qn], ref[b, :, :qn], f"{kind} seq {b}")
        assert torch.all(got[b, :, qn:] == sentinel)   # padding rows are not written
    lse_h = lse.cpu().numpy().reshape(B, Hq, q_len)
    for b in range(B):
        np.testing.assert_allclose(lse_h[b, :, :q_lens[b]], ref_lse[b, :, :q_lens[b]],
                                   rtol=0, atol=1e-4)


RAGGED_F32 = [
    # (B, Hq, Hkv, D, P, q_len, seq_lens, q_lens, call kwargs): the fp32 split kernel, whose
    # CTAs load their query rows before seq_len and q_lens are known
    (2, 8, 2, 128, 16, 3, [400, 90], [2, 3], {}),                      # cluster merge
    (2, 8, 2, 128, 16, 3, [400, 90], [2, 1], dict(split_tokens=64)),   # splits + merge kernel
    (3, 8, 4, 64, 16, 2, [300, 77, 500], [1, 2, 0], {}),
]


@pytest.mark.parametrize("B,Hq,Hkv,D,P,q_len,lens,q_lens,kw", RAGGED_F32)
def test_ragged_f32_with_poisoned_padding_rows(B, Hq, Hkv, D, P, q_len, lens, q_lens, kw):
    prob = inputs.make("suffix", B, Hq, Hkv, D, P, lens, q_len=q_len, dtype="f32",
                       seed=90 + q_len)
    for b in range(B):  # padding query rows hold NaN: masked if read, never written
        prob.q[b, :, q_lens[b]:, :] = float("nan")
    ref, ref_lse = oracle_rows(prob, want_lse=True, q_lens=np.int32(q_lens))
    dev = prob.to(DEV)
    ql = torch.tensor(q_lens, dtype=torch.int32, device=DEV)
    sentinel = 12345.0
    out = torch.full(prob.q.shape, sentinel, dtype=torch.float32, device=DEV)
    lse = torch.full((flat_rows(prob),), sentinel, dtype=torch.float32, device=DEV)
    status = torch.zeros(1, dtype=torch.int32, device=DEV)
    run_gpu(dev, out=out, out_dtype=torch.float32, lse=lse, status=status, q_lens=ql, **kw)
    torch.cuda.synchronize()
    assert int(status.item()) == 0
    got = out.cpu()
    lse_h = lse.cpu().numpy().reshape(B, Hq, q_len)
    for b in range(B):
        qn = q_lens[b]
        if qn:
            assert_parity(prob, got[b, :, :qn], ref[b, :, :qn], f"f32 ragged seq {b}")
            np.testing.assert_allclose(lse_h[b, :, :qn], ref_lse[b, :, :qn], rtol=0, atol=2e-5)
        assert torch.all(got[b, :, qn:] == sentinel)
        assert np.all(lse_h[b, :, qn:] == sentinel)
