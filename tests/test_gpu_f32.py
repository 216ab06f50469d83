"""fp32 K/V with many query rows per (sequence, kv head): the tensor-core kernel
that takes each fp32 product as three tf32 products (suffix, prefill), against the
oracle at max|err| <= 1e-5 max|ref|, in split, automatic and direct-output modes."""
import numpy as np
import pytest
import torch

import exact_causal_gqa_gb300 as atlas
import oracle
from exact_causal_gqa_gb300 import inputs
from tests.gpu_helpers import assert_parity, flat_rows, oracle_rows, run_gpu

pytestmark = pytest.mark.gpu
DEV = "cuda"


def make(kind, B, Hq, Hkv, D, P, lens, q_len, seed, **kw):
    host = inputs.make(kind, B, Hq, Hkv, D, P, list(lens), q_len=q_len, dtype="f32",
                       out_dtype="f32", seed=seed, device="cpu", **kw)
    dev = inputs.Problem(**{k: (v.to(DEV) if torch.is_tensor(v) else v)
                            for k, v in vars(host).items()})
    return host, dev


@pytest.mark.parametrize("D", [64, 128])
@pytest.mark.parametrize("kind,B,Hq,Hkv,P,lens,q_len", [
    ("suffix", 3, 16, 2, 16, (300, 2000, 5000), 16),   # 128 columns per kv head
    ("suffix", 2, 8, 2, 32, (64, 1500), 16),           # 64 columns: the smallest tile case
    ("suffix", 2, 32, 4, 16, (4096, 777), 40),          # 320 columns: three tiles, a partial one
    ("prefill", 2, 8, 2, 16, (640, 640), 640),         # q_len a multiple of the tile: heavy-first
    ("prefill", 1, 4, 1, 64, (200,), 200),              # ragged tail tile
])
def test_tensor_core_f32_matches_oracle(kind, B, Hq, Hkv, P, lens, q_len, D):
    host, dev = make(kind, B, Hq, Hkv, D, P, lens, q_len, seed=D + q_len)
    ref, ref_lse = oracle_rows(host, want_lse=True)
    for split, flags in ((0, 0), (512, 0), (0, atlas.DEBUG_TC_DIRECT)):
        lse = torch.empty(flat_rows(host), dtype=torch.float32, device=DEV)
        status = torch.zeros(1, dtype=torch.int32, device=DEV)
        out = run_gpu(dev, split_tokens=split, debug_flags=flags, lse=lse, status=status)
        torch.cuda.synchronize()
        assert int(status.item()) == 0
        assert_parity(host, out, ref, f"{kind} f32 split {split} flags {flags}")
        np.testing.assert_allclose(lse.cpu().numpy(), ref_lse.reshape(-1), rtol=0, atol=2e-5)


def test_threshold_between_the_f32_kernels():
    # 16 columns per kv head (the split kernel) and 17, 63, 64 (the tensor-core kernel)
    for Hq, q_len in ((8, 2), (17, 1), (9, 7), (8, 8)):
        host, dev = make("suffix", 2, Hq, 1, 128, 16, (900, 333), q_len, seed=Hq)
        out = run_gpu(dev)
        torch.cuda.synchronize()
        assert_parity(host, out, oracle_rows(host), f"{Hq}x{q_len} columns")


@pytest.mark.parametrize("variant", [dict(window=300), dict(softcap=20.0), "sinks", "ragged"])
def test_tensor_core_f32_variants(variant):
    host, dev = make("suffix", 3, 16, 2, 128, 16, (700, 1900, 260), 16, seed=41)
    kw, okw = {}, {}
    if variant == "sinks":
        sinks = (torch.randn(16, generator=torch.Generator().manual_seed(2)) * 2).float()
        kw["sinks"], okw["sinks"] = sinks.to(DEV), sinks.numpy().astype(np.float64)
    elif variant == "ragged":
        q_lens = torch.tensor([16, 5, 1], dtype=torch.int32)
        kw["q_lens"], okw["q_lens"] = q_lens.to(DEV), q_lens.numpy()
    else:
        kw, okw = variant, variant
    out = run_gpu(dev, split_tokens=256, **kw)
    torch.cuda.synchronize()
    ref = oracle_rows(host, **okw)
    if variant == "ragged":
        # rows past q_lens[b] are not queries: compare the real rows only
        keep = np.zeros(ref.shape[:3], dtype=bool)
        for b, n in enumerate([16, 5, 1]):
            keep[b, :, :n] = True
        got = out.cpu().numpy().reshape(ref.shape)[keep]
        assert np.abs(got - ref[keep]).max() <= 1e-5 * np.abs(ref[keep]).max()
    else:
        assert_parity(host, out, ref, str(variant))


def test_suffix_at_scale_sampled_rows():
    """The suffix workload's shape (B16, SQ16, contexts 4K-64K, 32/4 heads, P32) in
    fp32: sampled output rows against the oracle computed row by row."""
    host = inputs.make_config(4, device="cpu", dtype="f32", out_dtype="f32")
    dev = inputs.Problem(**{k: (v.to(DEV) if torch.is_tensor(v) else v)
                            for k, v in vars(host).items()})
    out = run_gpu(dev)
    torch.cuda.synchronize()
    rng = np.random.default_rng(4)
    rows = np.sort(rng.choice(flat_rows(host), size=96, replace=False))
    ref = oracle_rows(host, rows=rows)
    got = out.reshape(-1, host.head_dim)[torch.from_numpy(rows).to(DEV)]
    assert_parity(host, got, ref, "f32 suffix at scale (sampled)")


@pytest.mark.parametrize("scale", [-0.09, 0.0, 0.3])
@pytest.mark.parametrize("D", [64, 128])
def test_tensor_core_f32_any_finite_scale(scale, D):
    # S = -Q K^T with |scale| for negative scales (Q negated exactly); 0: uniform weights
    host, dev = make("suffix", 2, 32, 4, D, 32, (200, 1000), 16, seed=7, scale=scale)
    out = run_gpu(dev)
    torch.cuda.synchronize()
    assert_parity(host, out, oracle_rows(host), f"scale {scale}")
    host, dev = make("prefill", 1, 8, 2, D, 64, (384,), 384, seed=8, scale=scale)
    out = run_gpu(dev, debug_flags=atlas.DEBUG_TC_DIRECT)
    torch.cuda.synchronize()
    assert_parity(host, out, oracle_rows(host), f"prefill scale {scale}")


@pytest.mark.parametrize("flags,split", [(atlas.DEBUG_TC_DIRECT, 0), (0, 256)])
def test_tensor_core_f32_bad_page_and_seq_len(flags, split):
    host, dev = make("suffix", 3, 32, 4, 128, 32, (300, 400, 500), 16, seed=4)
    dev.page_table[1, 2] = -3
    dev.seq_lens[2] = 7  # fewer keys than query rows
    status = torch.zeros(1, dtype=torch.int32, device=DEV)
    out = run_gpu(dev, status=status, split_tokens=split, debug_flags=flags)
    torch.cuda.synchronize()
    st = int(status.item())
    assert st & atlas.DEV_BAD_PAGE and st & atlas.DEV_BAD_SEQLEN
    assert torch.isnan(out[1]).all() and torch.isnan(out[2]).all()
    assert torch.isfinite(out[0]).all()


def test_prefill_at_scale_sampled_rows():
    """The causal prefill workload's shape (2 x 8192 rows, 32 / 8 heads, P64) in fp32,
    direct output: every row of one (sequence, kv head) group's first q head and a
    spread of the others against the oracle."""
    host = inputs.make_config(5, device="cpu", dtype="f32", out_dtype="f32")
    dev = inputs.Problem(**{k: (v.to(DEV) if torch.is_tensor(v) else v)
                            for k, v in vars(host).items()})
    out = run_gpu(dev)
    torch.cuda.synchronize()
    S, H = host.q_len, host.n_q_heads
    rng = np.random.default_rng(5)
    rows = np.unique(np.concatenate([
        [(1 * H + 9) * S + i for i in range(S)],
        rng.choice(flat_rows(host), size=256, replace=False)]))
    ref = oracle_rows(host, rows=rows)
    got = out.reshape(-1, host.head_dim)[torch.from_numpy(rows).to(DEV)]
    assert_parity(host, got, ref, "f32 prefill at scale (sampled)")
